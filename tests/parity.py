"""Helpers shared by the GPU parity tests: oracle runs on sampled tokens and
the tolerance check of the layer's bf16 output.

Tolerance of the final bf16 streams: |gpu - oracle| <= max(2e-2, one bf16 step
at the oracle's value) element-wise, and relative L2 <= 5e-3.  The 2e-2 bound
is below one bf16 step for |out| >= 4 (a step there is 2^-5 = 0.03125), where
two correct implementations that sum in different orders can round to
neighbouring bf16 values; such elements may differ by that one step.  Gates:
|gpu - oracle| <= 1e-3.  Gathered rows: bit-exact."""
from __future__ import annotations

import numpy as np

from engram_hashed_gram_gb300 import synth
from oracle import engram_oracle as O

ABS_TOL = 2e-2
REL_L2_TOL = 5e-3
GATE_TOL = 1e-3


def bf16_step(v: np.ndarray) -> np.ndarray:
    """One bf16 step (ulp) at |v|: 2^(e-8) for |v| in [2^(e-1), 2^e)."""
    _, e = np.frexp(np.abs(v))
    return np.ldexp(1.0, np.maximum(e - 8, -133))


def weight_values(inp: synth.HostInputs) -> np.ndarray:
    """The projection weight as float64 [N, K]: bf16 bits, or the MXFP8 codes
    and scales (through the oracle's definition)."""
    if inp.wkv_scale is None:
        return O.bf16_value(inp.wkv)
    return O.mxfp8_weight(inp.wkv, inp.wkv_scale)


def kv_bound(e_bits, w_values, kv_ref_bits, K: int, splits: int = 8):
    """Per-element bound on |gpu kv - oracle kv|: one bf16 step at the oracle
    value plus the fp32 dot-product error bound gamma_n * sum_k |e_k W_jk|
    (Higham, "Accuracy and Stability of Numerical Algorithms", section 3.1),
    with n = K/16 accumulator additions of MMA partials (16 or 32 products
    each), 32 more for the partial itself, and the split-K additions (8, the
    largest number of K ranges any plan sums).
    w_values: the weight as float64 [N, K] (weight_values)."""
    n = K // 16 + 32 + splits
    u = 2.0 ** -24
    gamma = n * u / (1 - n * u)
    absdot = np.abs(O.bf16_value(e_bits)) @ np.abs(np.asarray(w_values, dtype=np.float64)).T
    return bf16_step(O.bf16_value(kv_ref_bits)) + gamma * absdot


def compare_out(gpu_bits, ref_bits):
    g = O.bf16_value(gpu_bits).ravel()
    r = O.bf16_value(ref_bits).ravel()
    assert g.shape == r.shape
    err = np.abs(g - r)
    bound = np.maximum(ABS_TOL, bf16_step(r))
    nrm = float(np.linalg.norm(r))
    rel = float(np.linalg.norm(g - r)) / (nrm if nrm > 0 else 1.0)
    return {
        "max_err": float(err.max()) if err.size else 0.0,
        "n_over_abs": int((err > ABS_TOL).sum()),
        "n_bad": int((err > bound).sum()),
        "rel_l2": rel,
        "frac_diff": float((err > 0).mean()) if err.size else 0.0,
        "ok": bool(np.all(err <= bound) and rel <= REL_L2_TOL),
    }


def assert_out_close(gpu_bits, ref_bits, what=""):
    s = compare_out(gpu_bits, ref_bits)
    assert s["ok"], f"{what}: {s}"
    return s


def assert_bits_equal_nan_aware(a, b, what=""):
    a = np.asarray(a, dtype=np.uint16)
    b = np.asarray(b, dtype=np.uint16)
    na = np.isnan(O.bf16_value(a))
    nb = np.isnan(O.bf16_value(b))
    assert np.array_equal(na, nb), f"{what}: NaN positions differ"
    bad = np.flatnonzero((a != b) & ~na)
    assert bad.size == 0, f"{what}: {bad.size} bit mismatches, first at {bad[:5]}: {a.ravel()[bad[:5]]} vs {b.ravel()[bad[:5]]}"


def check_layer(w: synth.Workload, inp: synth.HostInputs, tok: np.ndarray, gpu_out, gpu_gates, gpu_kv,
                what: str = ""):
    """Stage-wise parity of the sampled tokens `tok`; returns a summary dict.

    1. kv (projection) against the oracle's kv, element by element, within one
       bf16 step plus the fp32 dot-product error bound (kv_bound).
    2. gates and output against the oracle's gate and residual steps fed the
       GPU's own kv: gates within GATE_TOL, output within max(ABS_TOL, one bf16
       step) per element and REL_L2_TOL overall.  Same inputs, so this is the
       strict check of the gate and residual kernels.
    3. end to end against the oracle from the ids: relative L2 within
       REL_L2_TOL, and each gate / output element within its stage-2 tolerance
       plus the change the oracle itself shows between its own kv and the GPU's
       (the triangle inequality: the part of the difference that the bounded kv
       difference of step 1 causes through the exact gate).  Near dot = 0 the
       signed square root's slope sigma'(z)/(2 sqrt|dot|) amplifies that part,
       so it is reported (pairs with an end-to-end gate difference above
       GATE_TOL) and capped: at most 2% of the pairs, gate difference <= 0.05."""
    M = len(tok)
    hc, D = w.hc_mult, w.dim
    ref_out, ref_g, ref_kv = oracle_tokens(w, inp, tok)
    x = inp.x.reshape(w.M, hc, D)[tok]
    mask = None if inp.mask is None else inp.mask.reshape(w.M)[tok]
    gpu_out = np.asarray(gpu_out, dtype=np.uint16).reshape(M, hc, D)
    gpu_gates = np.asarray(gpu_gates, dtype=np.float64).reshape(M, hc)
    gpu_kv = np.asarray(gpu_kv, dtype=np.uint16).reshape(M, -1)
    # 1. projection
    bound = kv_bound(oracle_rows(w, inp, tok), weight_values(inp), ref_kv, w.K)
    kv_err = np.abs(O.bf16_value(gpu_kv) - O.bf16_value(ref_kv))
    far = kv_err > bound
    assert not far.any(), f"{what}: kv outside the bound at {np.argwhere(far)[:5].tolist()} ({far.sum()})"
    # 2. gate + residual on identical kv
    g_same = O.gates(gpu_kv, x, inp.q, inp.k, mask, w.eps)
    out_same = O.residual(gpu_kv, x, g_same, mask)
    gate_err_same = float(np.max(np.abs(gpu_gates - g_same)))
    assert gate_err_same <= GATE_TOL, f"{what}: gate error {gate_err_same} on identical kv"
    s2 = compare_out(gpu_out, out_same)
    assert s2["ok"], f"{what}: output vs oracle on identical kv: {s2}"
    # 3. end to end
    s3 = compare_out(gpu_out, ref_out)
    assert s3["rel_l2"] <= REL_L2_TOL, f"{what}: end-to-end rel L2 {s3}"
    gate_e2e = np.abs(gpu_gates - ref_g)
    gate_kv = np.abs(g_same - ref_g)
    assert np.all(gate_e2e <= GATE_TOL + gate_kv), f"{what}: end-to-end gate difference not explained by kv"
    g, r, rs = O.bf16_value(gpu_out), O.bf16_value(ref_out), O.bf16_value(out_same)
    out_bad = np.abs(g - r) > np.maximum(ABS_TOL, bf16_step(rs)) + np.abs(rs - r)
    assert not out_bad.any(), (f"{what}: end-to-end output difference not explained by kv at "
                               f"{np.argwhere(out_bad)[:5].tolist()}")
    amplified = gate_e2e > GATE_TOL
    assert amplified.mean() <= 0.02 and gate_e2e.max() <= 0.05, f"{what}: gate {gate_e2e.max()}"
    with np.errstate(divide="ignore", invalid="ignore"):
        z = np.log(ref_g) - np.log1p(-ref_g)
    return {"kv_frac_diff": float((kv_err > 0).mean()), "gate_err_same_kv": gate_err_same,
            "out_same_kv": s2, "end_to_end": s3, "gate_err_e2e": float(gate_e2e.max()),
            "pairs_gate_over_tol": int(amplified.sum()), "pairs": int(amplified.size),
            "min_abs_dot_of_those": float(np.min(z[amplified] ** 2)) if amplified.any() else None}


def compact_rows(w: synth.Workload, ids: np.ndarray, seed: int | None = None):
    """Regenerates only the table rows that `ids` reference (the full table may
    be ~100 GB) and remaps the ids onto that compact table; ids outside
    [0, R) stay outside it.  Returns (compact_ids, codes, scales)."""
    R = w.num_rows()
    seed = w.seed if seed is None else seed
    ids = np.asarray(ids, dtype=np.int64)
    valid = (ids >= 0) & (ids < R)
    uniq = np.unique(ids[valid])
    if uniq.size:
        codes, scales = synth.table_rows(seed, uniq, w.head_dim, w.scale_block, w.scale_fmt)
    else:
        codes = np.zeros((1, w.head_dim), np.uint8)
        nb = w.head_dim // w.scale_block
        scales = np.full((1, nb), 127, np.uint8) if w.scale_fmt == 1 else np.ones((1, nb), np.float32)
    out = np.full(ids.shape, -1, dtype=np.int64)
    out[valid] = np.searchsorted(uniq, ids[valid])
    return out, codes, scales


def oracle_rows(w: synth.Workload, inp: synth.HostInputs, tok: np.ndarray) -> np.ndarray:
    """Oracle gathered rows (bf16 bits [n, K]) of the tokens `tok`."""
    ids = inp.hash_ids.reshape(w.M, w.n_cols)[tok]
    cids, codes, scales = compact_rows(w, ids)
    return O.lookup(cids, codes, scales, w.scale_block, w.scale_fmt)


def oracle_tokens(w: synth.Workload, inp: synth.HostInputs, tok: np.ndarray, eps: float | None = None):
    """Oracle (out bits [n, hc, dim], gates [n, hc], kv bits [n, N]) for the
    tokens `tok` (flat indices into B*T) of a workload."""
    M = w.M
    ids = inp.hash_ids.reshape(M, w.n_cols)[tok]
    cids, codes, scales = compact_rows(w, ids)
    x = inp.x.reshape(M, w.hc_mult, w.dim)[tok]
    mask = None if inp.mask is None else inp.mask.reshape(M)[tok]
    return O.forward(cids, x, codes, scales, inp.wkv, inp.q, inp.k, mask, scale_block=w.scale_block,
                     scale_fmt=w.scale_fmt, eps=w.eps if eps is None else eps, wkv_scale=inp.wkv_scale)


def sample_tokens(M: int, n: int, rng, must=()) -> np.ndarray:
    """n token indices: the first and last, the given ones, and uniform draws."""
    pick = {0, M - 1, *[int(m) for m in must if 0 <= m < M]}
    if M > len(pick):
        extra = rng.choice(M, size=min(M, n) , replace=False)
        for e in extra:
            if len(pick) >= n:
                break
            pick.add(int(e))
    return np.array(sorted(pick), dtype=np.int64)
