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
        codes, scales = synth.table_rows(seed, uniq, w.head_dim, w.scale_block)
    else:
        codes = np.zeros((1, w.head_dim), np.uint8)
        scales = np.ones((1, w.head_dim // w.scale_block), np.float32)
    out = np.full(ids.shape, -1, dtype=np.int64)
    out[valid] = np.searchsorted(uniq, ids[valid])
    return out, codes, scales


def oracle_tokens(w: synth.Workload, inp: synth.HostInputs, tok: np.ndarray, eps: float | None = None):
    """Oracle (out bits [n, hc, dim], gates [n, hc], kv bits [n, N]) for the
    tokens `tok` (flat indices into B*T) of a workload."""
    M = w.M
    ids = inp.hash_ids.reshape(M, w.n_cols)[tok]
    cids, codes, scales = compact_rows(w, ids)
    x = inp.x.reshape(M, w.hc_mult, w.dim)[tok]
    mask = None if inp.mask is None else inp.mask.reshape(M)[tok]
    return O.forward(cids, x, codes, scales, inp.wkv, inp.q, inp.k, mask, scale_block=w.scale_block,
                     eps=w.eps if eps is None else eps)


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
