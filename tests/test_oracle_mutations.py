"""Plants plausible mistakes in the oracle (on the CPU, one at a time) and
checks that at least one pin of tests/test_oracle_pins.py fails for each, so
the pins are known to constrain every step."""
import numpy as np
import pytest

import test_oracle_pins as P
from oracle import engram_oracle as O

_orig_gates = O.gates
_orig_residual = O.residual
_orig_dequant = O.dequant_rows
_orig_lookup = O.lookup
_orig_mxfp8_weight = O.mxfp8_weight


def _gates_variant(no_dim_scale=False, joint=False, no_clamp=False, q_only=False,
                   eps_outside=False, sum_not_mean=False, no_sign=False):
    def g(kv_bits, x_bits, q_bits, k_bits, mask=None, eps=1e-6, clamp=1e-6):
        x = O.bf16_value(x_bits)
        M, S, D = x.shape
        kv = O.bf16_value(kv_bits).reshape(M, -1)
        key = kv[:, :S * D].reshape(M, S, D)
        w = O.bf16_value(q_bits).reshape(S, D)
        if not q_only:
            w = w * O.bf16_value(k_bits).reshape(S, D)
        red = np.sum if sum_not_mean else np.mean
        if joint:
            mh = np.repeat(red(x * x, axis=(-1, -2))[:, None] / S, S, axis=1)
        else:
            mh = red(x * x, axis=-1)
        mk = red(key * key, axis=-1)
        if eps_outside:
            rstd = 1.0 / np.sqrt(mh) / np.sqrt(mk) + eps
        else:
            rstd = (1.0 / np.sqrt(mh + eps)) * (1.0 / np.sqrt(mk + eps))
        dot = np.sum(x * w[None] * key, axis=-1) * rstd
        if not no_dim_scale:
            dot = dot * float(D) ** -0.5
        mag = np.abs(dot) if no_clamp else np.maximum(np.abs(dot), clamp)
        z = np.sqrt(mag) if no_sign else np.copysign(np.sqrt(mag), dot)
        out = 1.0 / (1.0 + np.exp(-z))
        if mask is not None:
            out = np.where(np.asarray(mask).reshape(M, 1).astype(bool), out, 0.0)
        return out
    return g


def _residual_first_block(kv_bits, x_bits, g, mask=None):
    xb = np.asarray(x_bits, dtype=np.uint16)
    M, S, D = xb.shape
    kv = O.bf16_value(kv_bits).reshape(M, -1)
    return O.round_to_bf16(O.bf16_value(xb) + g[:, :, None] * kv[:, None, :D])


def _residual_add_even_if_masked(kv_bits, x_bits, g, mask=None):
    return _orig_residual(kv_bits, x_bits, g, None)


def _dequant_wrong_block(codes, scales, scale_block, scale_fmt=O.SCALE_F32):
    codes = np.asarray(codes, dtype=np.uint8)
    n, hd = codes.shape
    nb = hd // scale_block
    v = O.decode_e4m3(codes).astype(np.float32)
    s = np.asarray(scales, dtype=np.float32).reshape(n, nb)
    idx = np.arange(hd) % nb                                   # interleaved instead of blocked
    return O.round_to_bf16((v * s[:, idx]).astype(np.float64))


def _dequant_double_product(codes, scales, scale_block, scale_fmt=O.SCALE_F32):
    codes = np.asarray(codes, dtype=np.uint8)
    n, hd = codes.shape
    v = O.decode_e4m3(codes)
    s = np.asarray(scales, dtype=np.float64).reshape(n, hd // scale_block)
    return O.round_to_bf16((v.reshape(n, -1, scale_block) * s[:, :, None]).reshape(n, hd))


def _lookup_transposed(hash_ids, table, scale, scale_block, scale_fmt=O.SCALE_F32):
    e = _orig_lookup(hash_ids, table, scale, scale_block, scale_fmt)
    M, C = np.asarray(hash_ids).shape
    hd = np.asarray(table).shape[1]
    return e.reshape(M, C, hd).transpose(0, 2, 1).reshape(M, C * hd)


def _mxfp8_block_64(codes, scales, block=32):
    c = np.asarray(codes, dtype=np.uint8)
    N, K = c.shape
    s = O.decode_e8m0(np.asarray(scales, dtype=np.uint8).reshape(N, -1))
    idx = np.minimum(np.arange(K) // 64, s.shape[1] - 1)          # one scale per 64 inputs
    return O.decode_e4m3(c) * s[:, idx]


def _mxfp8_scale_interleaved(codes, scales, block=32):
    c = np.asarray(codes, dtype=np.uint8)
    N, K = c.shape
    s = O.decode_e8m0(np.asarray(scales, dtype=np.uint8).reshape(N, -1))
    return O.decode_e4m3(c) * s[:, np.arange(K) % s.shape[1]]


def _mxfp8_no_bias(codes, scales, block=32):
    c = np.asarray(codes, dtype=np.uint8)
    N, K = c.shape
    s = np.ldexp(1.0, np.asarray(scales, dtype=np.int64).reshape(N, -1) - 126)   # bias off by one
    return O.decode_e4m3(c) * s[:, np.arange(K) // block]


def _round_truncate(x):
    x = np.asarray(x, dtype=np.float64)
    return (x.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


MUTATIONS = {
    "gate: no dim^-0.5": ("gates", _gates_variant(no_dim_scale=True)),
    "gate: joint normalisation": ("gates", _gates_variant(joint=True)),
    "gate: no clamp": ("gates", _gates_variant(no_clamp=True)),
    "gate: q only": ("gates", _gates_variant(q_only=True)),
    "gate: eps outside rsqrt": ("gates", _gates_variant(eps_outside=True)),
    "gate: sum not mean": ("gates", _gates_variant(sum_not_mean=True)),
    "gate: sign dropped": ("gates", _gates_variant(no_sign=True)),
    "residual: value from first block": ("residual", _residual_first_block),
    "residual: add on masked tokens": ("residual", _residual_add_even_if_masked),
    "dequant: wrong scale block": ("dequant_rows", _dequant_wrong_block),
    "dequant: product not rounded to fp32": ("dequant_rows", _dequant_double_product),
    "lookup: transposed flatten": ("lookup", _lookup_transposed),
    "bf16: truncation": ("round_to_bf16", _round_truncate),
    "mxfp8 weight: one scale per 64": ("mxfp8_weight", _mxfp8_block_64),
    "mxfp8 weight: scales interleaved": ("mxfp8_weight", _mxfp8_scale_interleaved),
    "mxfp8 weight: E8M0 bias off by one": ("mxfp8_weight", _mxfp8_no_bias),
}

PINS = [getattr(P, n) for n in dir(P) if n.startswith("test_") and n != "test_forward_tiny_vs_torch_restatement"]


def _run_pin(fn):
    import inspect
    params = inspect.signature(fn).parameters
    if "scale_block" in params:
        for sb in (128, 32, 256):
            fn(sb)
    else:
        fn()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_some_pin_catches_mutation(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(O, attr, fn)
    caught = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                _run_pin(pin)
        except Exception:
            caught.append(pin.__name__)
    assert caught, f"no pin fails under mutation {name!r}"
