"""Pins of the CPU oracle against facts fixed outside it: values the pages
print, closed forms, library routines for the number formats, and brute force
on tiny inputs.  Each test is chosen so that a plausible slip in the oracle (a
dropped term, a wrong sign or index, a transposed operand) fails it."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import read_golden
from engram_hashed_gram_gb300 import synth
from oracle import engram_oracle as O


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits(a) -> np.ndarray:
    return bits_of(torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16))


# ---------------------------------------------------------------------------
# printed values: parameter count and row layout
# ---------------------------------------------------------------------------
def test_parameter_count_matches_page_table():
    g = read_golden("engram_parameters.txt")
    rows = g["instance_rows"]
    total = O.parameter_count(rows, g["head_dim"], 24, g["dim"], g["hc_mult"])
    assert total == g["instance_params"] == 98_465_597_952
    assert rows * g["head_dim"] == g["table_params"]
    assert (3 * 8 * g["head_dim"]) * (g["dim"] * (g["hc_mult"] + 1)) == g["wkv_params"]
    assert 2 * g["hc_mult"] * g["dim"] == g["gate_params"]
    assert 24 * g["head_dim"] == g["wkv_in"] and g["dim"] * (g["hc_mult"] + 1) == g["wkv_out"]


def test_prime_row_ranges_match_config():
    g = read_golden("engram_parameters.txt")
    n_cols = (g["engram_max_ngram_size"] - 1) * g["engram_n_heads"]
    primes = synth.consecutive_primes_above(g["engram_vocab_size"], 2 * n_cols)
    assert primes[0] == g["first_prime_module_0"]
    assert sum(primes[:n_cols]) == g["engram_num_embeddings_0"]
    assert sum(primes[n_cols:]) == g["engram_num_embeddings_1"]
    lengths, offsets = synth.workload("full_2x8192").layout()
    assert int(lengths.sum()) == g["instance_rows"]
    assert offsets[0] == 0 and all(offsets[c + 1] == offsets[c] + lengths[c] for c in range(n_cols - 1))


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------
def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.decode_e4m3(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_e4m3_decode_named_values():
    d = lambda c: float(O.decode_e4m3(np.array([c], dtype=np.uint8))[0])
    assert d(0x38) == 1.0
    assert d(0x7E) == 448.0 and d(0xFE) == -448.0
    assert d(0x08) == 2.0 ** -6           # smallest normal
    assert d(0x01) == 2.0 ** -9           # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9       # largest subnormal
    assert d(0x40) == 2.0 and d(0x3C) == 1.5
    assert d(0x80) == 0.0 and math.copysign(1.0, d(0x80)) == -1.0
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))


def test_e8m0_decode():
    d = O.decode_e8m0(np.array([127, 0, 254, 255, 130], dtype=np.uint8))
    assert d[0] == 1.0 and d[1] == 2.0 ** -127 and d[2] == 2.0 ** 127
    assert math.isnan(d[3]) and d[4] == 8.0


def test_round_to_bf16_matches_torch_on_fp32():
    rng = np.random.default_rng(0)
    n = 400_000
    mant = rng.integers(0, 1 << 23, size=n, dtype=np.uint32)
    exp = rng.integers(0, 255, size=n, dtype=np.uint32)      # includes subnormals, no inf/nan
    sign = rng.integers(0, 2, size=n, dtype=np.uint32)
    # force a third of the samples onto exact ties (low 16 bits = 0x8000)
    tie = rng.random(n) < 0.33
    mant = np.where(tie, (mant & ~np.uint32(0xFFFF)) | np.uint32(0x8000), mant)
    u = (sign << np.uint32(31)) | (exp << np.uint32(23)) | mant
    f = u.view(np.float32)
    ref = bits_of(torch.from_numpy(f.copy()).to(torch.bfloat16))
    got = O.round_to_bf16(f.astype(np.float64))
    assert np.array_equal(got, ref)


def test_round_to_bf16_rounds_once_from_float64():
    one = 1.0
    cases = [
        (one + 2.0 ** -8, 0x3F80),                 # tie -> even (1.0)
        (one + 3 * 2.0 ** -8, 0x3F82),             # tie -> even (1 + 2^-6)
        (one + 2.0 ** -8 + 2.0 ** -30, 0x3F81),    # just above the tie: up (an fp32 detour would give 1.0)
        (-(one + 2.0 ** -8 + 2.0 ** -30), 0xBF81),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (2.0 ** -133, 0x0001),                     # smallest bf16 subnormal
        (2.0 ** -134, 0x0000),                     # half of it: tie -> even (zero)
        (3.0e38, 0x7F62),
        (3.5e38, 0x7F80),                          # past the largest finite bf16
        (float("inf"), 0x7F80),
        (float("-inf"), 0xFF80),
    ]
    for x, want in cases:
        got = int(O.round_to_bf16(np.array([x]))[0])
        assert got == want, (x, hex(got), hex(want))
    assert (int(O.round_to_bf16(np.array([np.nan]))[0]) & 0x7FFF) > 0x7F80


# ---------------------------------------------------------------------------
# a2-a3: gather and dequantisation, brute force on a tiny table
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("scale_block", [128, 32, 256])
def test_dequant_all_codes_vs_library(scale_block):
    rng = np.random.default_rng(scale_block)
    R, hd = 29, 256
    codes = np.stack([rng.permutation(256).astype(np.uint8) for _ in range(R)])
    nb = hd // scale_block
    scales = np.exp(rng.normal(0.0, 0.5, size=(R, nb))).astype(np.float32)
    scales[0, :] = 1.0
    scales[1, :] = 0.125
    scales[2, :] = 32.0
    scales[3, :] = np.float32(1.0 / 3.0)
    got = O.dequant_rows(codes, scales, scale_block)
    # the excerpt's two lines, restated with torch's own fp8 widening and casts
    v = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float()
    s = torch.from_numpy(scales.copy())
    ref = (v.unflatten(-1, (-1, scale_block)) * s.unsqueeze(-1)).flatten(-2).to(torch.bfloat16)
    refb = bits_of(ref)
    nan = np.isnan(O.bf16_value(refb))
    assert np.array_equal(np.isnan(O.bf16_value(got)), nan)
    assert np.array_equal(got[~nan], refb[~nan])


def test_dequant_e8m0_scales():
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 256, size=(7, 256)).astype(np.uint8)
    codes[codes == 0x7F] = 0x7E
    codes[codes == 0xFF] = 0xFE
    sc = rng.integers(117, 137, size=(7, 8)).astype(np.uint8)
    got = O.bf16_value(O.dequant_rows(codes, sc, 32, O.SCALE_E8M0))
    v = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    s = np.ldexp(1.0, sc.astype(np.int64) - 127)
    ref = (v.reshape(7, 8, 32) * s[:, :, None]).reshape(7, 256)   # powers of two: exact
    assert np.array_equal(got, ref)


def test_lookup_layout_and_out_of_range_rows():
    rng = np.random.default_rng(7)
    R, hd, C, M = 13, 64, 5, 6
    codes = rng.integers(0, 0x7E, size=(R, hd)).astype(np.uint8)   # positive, finite
    scales = (1.0 + np.arange(R * 2, dtype=np.float32).reshape(R, 2))
    ids = rng.integers(0, R, size=(M, C))
    ids[0, 0] = -1
    ids[1, 3] = R
    ids[2, 4] = R + 1000
    ids[3, 1] = np.iinfo(np.int64).min
    e = O.bf16_value(O.lookup(ids, codes, scales, 32)).reshape(M, C, hd)
    vals = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    for m in range(M):
        for c in range(C):
            r = int(ids[m, c])
            for f in range(hd):
                if 0 <= r < R:
                    want = float(np.float32(vals[r, f]) * scales[r, f // 32])
                    want_b = O.bf16_value(bf16_bits([want]))[0]
                    assert e[m, c, f] == want_b
                else:
                    assert e[m, c, f] == 0.0 and not math.copysign(1.0, e[m, c, f]) < 0


# ---------------------------------------------------------------------------
# a4: projection
# ---------------------------------------------------------------------------
def test_project_identity_like_weight_copies_inputs():
    rng = np.random.default_rng(1)
    M, K, N = 5, 96, 160
    e = bf16_bits(rng.standard_normal((M, K)))
    perm = (7 * np.arange(N) + 3) % K
    W = np.zeros((N, K), dtype=np.float32)
    W[np.arange(N), perm] = 1.0
    kv = O.project(e, bf16_bits(W))
    assert np.array_equal(kv, e[:, perm])


def test_project_brute_force_exact_sums():
    rng = np.random.default_rng(2)
    M, K, N = 3, 40, 17
    e = bf16_bits(rng.standard_normal((M, K)))
    W = bf16_bits(rng.standard_normal((N, K)) * 0.3)
    kv = O.bf16_value(O.project(e, W))
    ev, wv = O.bf16_value(e), O.bf16_value(W)
    for m in range(M):
        for j in range(N):
            exact = sum((Fraction(float(ev[m, k])) * Fraction(float(wv[j, k])) for k in range(K)), Fraction(0))
            got = Fraction(float(kv[m, j]))
            # the result is the bf16 value nearest to the exact sum
            x = float(exact)
            _, ex = math.frexp(x)
            ulp = Fraction(2) ** (ex - 8)
            assert abs(got - exact) <= ulp / 2
            assert Fraction(float(got)) / ulp == int(Fraction(float(got)) / ulp)


def _e4m3_library(codes):
    """e4m3 codes -> float64 through torch's float8_e4m3fn widening."""
    c = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return c.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_mxfp8_weight_identity_copies_inputs():
    """One 1.0 per output row (code 0x38, scale 2^0) makes the FP8 projection
    a bit-exact copy of the chosen input channels; a scale one step up doubles
    every value exactly."""
    rng = np.random.default_rng(11)
    M, K, N = 4, 128, 96
    e = bf16_bits(rng.standard_normal((M, K)))
    perm = (5 * np.arange(N) + 1) % K
    codes = np.zeros((N, K), dtype=np.uint8)
    codes[np.arange(N), perm] = 0x38
    scales = np.full((N, K // 32), 127, dtype=np.uint8)
    assert np.array_equal(O.project_mxfp8(e, codes, scales), e[:, perm])
    up = O.bf16_value(O.project_mxfp8(e, codes, scales + 1))
    assert np.array_equal(up, 2.0 * O.bf16_value(e[:, perm]))


def test_mxfp8_block_scales_closed_form():
    """All-ones input and weight codes 1.0 with scale 2^(b mod 5 - 2) on block
    b: kv = 32 * sum_b 2^(b mod 5 - 2), one scale per 32 consecutive inputs."""
    K, N = 320, 7
    e = bf16_bits(np.ones((1, K)))
    codes = np.full((N, K), 0x38, dtype=np.uint8)
    nb = K // 32
    scales = np.tile((127 + (np.arange(nb) % 5) - 2).astype(np.uint8), (N, 1))
    scales[3] = 127                                             # one row unscaled
    kv = O.bf16_value(O.project_mxfp8(e, codes, scales))
    want = 32 * sum(2.0 ** ((b % 5) - 2) for b in range(nb))
    assert np.all(kv[0, [0, 1, 2, 4, 5, 6]] == want)
    assert kv[0, 3] == 32 * nb


def test_mxfp8_projection_brute_force():
    """Random codes (both signs, subnormals included) and scales against exact
    rational sums of torch-widened codes times 2^(s-127), rounded once."""
    rng = np.random.default_rng(12)
    M, K, N = 3, 96, 11
    e = bf16_bits(rng.standard_normal((M, K)))
    codes = rng.integers(0, 256, size=(N, K)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3A                       # no NaN codes
    scales = rng.integers(120, 134, size=(N, K // 32)).astype(np.uint8)
    kv = O.bf16_value(O.project_mxfp8(e, codes, scales))
    ev = O.bf16_value(e)
    wv = _e4m3_library(codes)
    for m in range(M):
        for j in range(N):
            exact = sum((Fraction(float(ev[m, k])) * Fraction(float(wv[j, k]))
                         * Fraction(2) ** (int(scales[j, k // 32]) - 127) for k in range(K)), Fraction(0))
            got = Fraction(float(kv[m, j]))
            x = float(exact)
            if x == 0.0:
                assert got == 0
                continue
            _, ex = math.frexp(x)
            ulp = Fraction(2) ** (ex - 8)
            assert abs(got - exact) <= ulp / 2


# ---------------------------------------------------------------------------
# a6-a7: gate
# ---------------------------------------------------------------------------
def _kv_from(key, value):
    """kv bits [M, S*D + D] from float arrays key [M, S, D] and value [M, D]."""
    M, S, D = key.shape
    return bf16_bits(np.concatenate([key.reshape(M, S * D), value], axis=1))


def _ones(S, D):
    return bf16_bits(np.ones((S, D)))


def sigmoid(z):
    return 1.0 / (1.0 + math.exp(-z))


def test_gate_dot_zero_gives_sigmoid_of_clamp_root():
    rng = np.random.default_rng(3)
    M, S, D = 4, 4, 5120
    x = bf16_bits(rng.standard_normal((M, S, D)))
    kv = _kv_from(np.zeros((M, S, D)), rng.standard_normal((M, D)))
    g = O.gates(kv, x, _ones(S, D), _ones(S, D))
    assert np.allclose(g, sigmoid(1e-3), rtol=0, atol=1e-15)
    assert abs(sigmoid(1e-3) - 0.500249999979167) < 1e-14


def test_gate_key_parallel_to_stream():
    """key = c*h with q = k = 1 and eps = 0: rstd = 1/(|c| mean h^2), so
    dot = sign(c) * sqrt(D) and gate = sigmoid(sign(c) * D^(1/4))."""
    rng = np.random.default_rng(4)
    M, S, D = 3, 4, 5120
    h = O.bf16_value(bf16_bits(rng.standard_normal((M, S, D))))
    for c, sgn in ((2.0, 1.0), (-2.0, -1.0), (0.25, 1.0)):
        kv = _kv_from(c * h, np.zeros((M, D)))
        g = O.gates(kv, bf16_bits(h), _ones(S, D), _ones(S, D), eps=0.0)
        assert np.allclose(g, sigmoid(sgn * D ** 0.25), rtol=0, atol=1e-12)
    assert abs(sigmoid(D ** 0.25) - 0.999788054644871) < 1e-12


def test_gate_uses_product_of_q_and_k_weights():
    """q = 2, k = 1.5 scales h*w*key by 3: dot = 3*sqrt(D)."""
    rng = np.random.default_rng(5)
    M, S, D = 2, 4, 1024
    h = O.bf16_value(bf16_bits(rng.standard_normal((M, S, D))))
    kv = _kv_from(h, np.zeros((M, D)))
    q = bf16_bits(np.full((S, D), 2.0))
    k = bf16_bits(np.full((S, D), 1.5))
    g = O.gates(kv, bf16_bits(h), q, k, eps=0.0)
    assert np.allclose(g, sigmoid(math.sqrt(3 * math.sqrt(D))), rtol=0, atol=1e-12)


def test_gate_odd_symmetry():
    rng = np.random.default_rng(6)
    M, S, D = 8, 4, 5120
    x = bf16_bits(rng.standard_normal((M, S, D)))
    key = rng.standard_normal((M, S, D))
    q, k = synth.make_qk(synth.workload(0))
    gp = O.gates(_kv_from(key, np.zeros((M, D))), x, q, k)
    gm = O.gates(_kv_from(-key, np.zeros((M, D))), x, q, k)
    assert np.allclose(gp + gm, 1.0, rtol=0, atol=1e-13)
    assert np.all(np.abs(gp - 0.5) > 1e-6)


def test_gate_normalised_per_stream_not_jointly():
    """Scaling one stream of h by 64 leaves every gate unchanged (eps = 0);
    normalising over all streams jointly would move the others."""
    rng = np.random.default_rng(8)
    M, S, D = 3, 4, 2048
    h = O.bf16_value(bf16_bits(rng.standard_normal((M, S, D))))
    key = rng.standard_normal((M, S, D))
    kv = _kv_from(key, np.zeros((M, D)))
    g0 = O.gates(kv, bf16_bits(h), _ones(S, D), _ones(S, D), eps=0.0)
    h2 = h.copy()
    h2[:, 0] *= 64.0
    g1 = O.gates(kv, bf16_bits(h2), _ones(S, D), _ones(S, D), eps=0.0)
    assert np.allclose(g0, g1, rtol=0, atol=1e-13)
    # and the streams are paired with their own key block: permuting both permutes the gates
    perm = [2, 0, 3, 1]
    kvp = _kv_from(O.bf16_value(kv)[:, :S * D].reshape(M, S, D)[:, perm], np.zeros((M, D)))
    gp = O.gates(kvp, bf16_bits(h[:, perm]), _ones(S, D), _ones(S, D), eps=0.0)
    assert np.allclose(gp, g0[:, perm], rtol=0, atol=1e-13)


def test_gate_eps_with_constant_vectors():
    """h = a and key = b constant, w = 1:
    dot = sqrt(D) * a * b / sqrt((a^2 + eps) (b^2 + eps))."""
    M, S, D = 1, 4, 5120
    a, b, eps = 2.0 ** -13, 0.5, 1e-6
    h = np.full((M, S, D), a)
    key = np.full((M, S, D), b)
    kv = _kv_from(key, np.zeros((M, D)))
    g = O.gates(kv, bf16_bits(h), _ones(S, D), _ones(S, D), eps=eps)
    dot = math.sqrt(D) * a * b / math.sqrt((a * a + eps) * (b * b + eps))
    assert 0 < dot < 0.2 * math.sqrt(D)      # eps dominates mean h^2 here
    assert np.allclose(g, sigmoid(math.sqrt(dot)), rtol=0, atol=1e-12)
    # eps = 1e-20 (the model config's norm_eps) gives dot ~ sqrt(D)
    g20 = O.gates(kv, bf16_bits(h), _ones(S, D), _ones(S, D), eps=1e-20)
    assert np.allclose(g20, sigmoid(D ** 0.25), rtol=0, atol=1e-9)


# ---------------------------------------------------------------------------
# a8: residual add and the mask
# ---------------------------------------------------------------------------
def test_value_is_the_last_block_and_shared_by_streams():
    rng = np.random.default_rng(9)
    M, S, D = 3, 2, 8
    h = rng.standard_normal((M, S, D))
    key = np.zeros((M, S, D))
    key[:, 0, :] = 1000.0               # a slip that reads a key block as the value shows up
    value = rng.standard_normal((M, D)) * 4
    kv = _kv_from(key, value)
    xb = bf16_bits(h)
    g = np.full((M, S), 0.75)
    out = O.bf16_value(O.residual(kv, xb, g))
    hv, vv = O.bf16_value(xb), O.bf16_value(bf16_bits(value))
    for m in range(M):
        for s in range(S):
            for d in range(D):
                exact = hv[m, s, d] + 0.75 * vv[m, d]        # exact in float64 here
                want = O.bf16_value(O.round_to_bf16(np.array([exact])))[0]
                assert out[m, s, d] == want


def test_mask_false_passes_bits_through():
    rng = np.random.default_rng(10)
    M, S, D = 6, 4, 256
    xf = rng.standard_normal((M, S, D)).astype(np.float32)
    xf[1, 2, :7] = -0.0
    x = bf16_bits(xf)
    kv = _kv_from(rng.standard_normal((M, S, D)), rng.standard_normal((M, D)))
    kv = kv.copy()
    kv[1, S * D + 3] = 0x7F80      # +inf in the value of a masked token
    kv[4, S * D + 5] = 0x7FC0      # NaN in the value of a masked token
    mask = np.array([1, 0, 1, 1, 0, 1], dtype=np.uint8)
    g = O.gates(kv, x, _ones(S, D), _ones(S, D), mask)
    out = O.residual(kv, x, g, mask)
    assert np.array_equal(out[~mask.astype(bool)], x[~mask.astype(bool)])
    assert np.all(g[~mask.astype(bool)] == 0.0)
    assert not np.array_equal(out[mask.astype(bool)], x[mask.astype(bool)])


def test_forward_tiny_vs_torch_restatement():
    """Cross-check of the assembled layer on a tiny shape against the excerpt
    run with torch CPU ops in the excerpt's own fp32 (not a pin by itself: the
    pins above fix each step)."""
    rng = np.random.default_rng(11)
    M, S, D, C, hd, R = 5, 4, 256, 3, 64, 50
    codes = rng.integers(0, 0x7E, size=(R, hd)).astype(np.uint8)
    codes[rng.random((R, hd)) < 0.5] |= 0x80
    scales = np.exp(rng.normal(0, 0.5, size=(R, hd // 32))).astype(np.float32)
    ids = rng.integers(0, R, size=(M, C))
    ids[0, 1] = R + 3
    W = bf16_bits(rng.standard_normal((D * (S + 1), C * hd)) / math.sqrt(C * hd))
    q = bf16_bits(1 + 0.3 * rng.standard_normal((S, D)))
    k = bf16_bits(1 + 0.3 * rng.standard_normal((S, D)))
    x = bf16_bits(rng.standard_normal((M, S, D)))
    mask = np.array([1, 1, 0, 1, 1], dtype=np.uint8)
    out, g, kv = O.forward(ids, x, codes, scales, W, q, k, mask, scale_block=32)

    t = lambda b: torch.from_numpy(b.astype(np.int16)).view(torch.bfloat16)
    idx = torch.from_numpy(ids)
    valid = (idx >= 0) & (idx < R)
    li = idx.masked_fill(~valid, 0)
    vals = torch.from_numpy(codes)[li].view(torch.float8_e4m3fn).float()
    sc = torch.from_numpy(scales)[li]
    e = (vals.unflatten(-1, (-1, 32)) * sc.unsqueeze(-1)).flatten(-2).to(torch.bfloat16)
    e = e.masked_fill(~valid.unsqueeze(-1), 0).flatten(-2)
    kvt = (e.float() @ t(W).float().T).to(torch.bfloat16)
    key, value = kvt.split([S * D, D], dim=-1)
    key = key.float().unflatten(-1, (S, D))
    wt = t(q).float() * t(k).float()
    h = t(x).float()
    rstd = torch.rsqrt(h.square().mean(-1) + 1e-6) * torch.rsqrt(key.square().mean(-1) + 1e-6)
    dot = (h * wt * key).sum(-1) * rstd * D ** -0.5
    gt = torch.sigmoid(torch.copysign(dot.abs().clamp_min(1e-6).sqrt(), dot))
    mt = torch.from_numpy(mask.astype(bool))
    gt = gt.masked_fill(~mt.unsqueeze(-1), 0)
    ot = (h + gt.unsqueeze(-1) * value.float().unsqueeze(-2)).to(torch.bfloat16)
    ot = torch.where(mt.view(M, 1, 1), ot, t(x))

    kv_diff = np.abs(O.bf16_value(kv) - kvt.double().numpy())
    assert np.mean(kv_diff > 0) < 0.01
    assert np.max(np.abs(g - gt.double().numpy())) < 1e-5
    od = np.abs(O.bf16_value(out) - ot.double().numpy())
    assert od.max() <= 2.0 ** -4 and np.mean(od > 0) < 0.01
