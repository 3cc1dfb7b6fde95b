"""CPU oracle for the Engram layer forward -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm may import this module.  The product path (the CUDA
library and its Python binding) never imports, links or calls it, and shares no
code with it.

What it computes, step by step, is the Engram layer of DeepSeek-V4.1-Flash as
printed in the code excerpts of atlas.klimoza.dev "deepseek-v4.1 /
engram-second" (the ``Engram`` class and the ``ParallelEngramEmbedding``
class), with the reading of the prose on zhuai.tech "Engram in DeepSeek V4.1
Flash" (section "Step 3: Inject memory at the correct layer boundary").

Precision.  The excerpts fix the precision of three steps and the oracle keeps
them: the dequantising multiply is an fp32 product of the widened code and the
fp32 scale, then a cast to bf16 (``ParallelEngramEmbedding.forward``); the
projection ``wkv`` returns the activation dtype, bf16; the layer returns
``x.dtype``, bf16.  Everything else (the projection's accumulation, the gate's
reductions and the residual add) is evaluated in float64 and rounded once, to
bf16, where the excerpt casts.  The result is the exact value of the excerpt's
formula up to that final rounding.  Rounding to bf16 is round-to-nearest-even,
written out below from its definition.

Readings where the pages leave a step open (each is also listed in the design
notes of the repository):
  * masked tokens (``token_mask`` False) return the input bits unchanged: the
    excerpt's docstring says such positions are left as they are; a literal
    ``h + 0*value`` would differ only for h = -0.0 or a non-finite value.
  * ids outside [0, R) give a zero row, as the single-rank case of the sharded
    embedding does (its out-of-shard mask zeroes the row).
  * eps is a parameter (the benchmark uses 1e-6; the model config's norm_eps is
    1e-20); clamp is the excerpt's ``clamp_value`` = 1e-6.

Parity pins live in ``tests/test_oracle_pins.py``.  No function here is
"parity unpinned".
"""
from __future__ import annotations

import numpy as np

SCALE_F32 = 0
SCALE_E8M0 = 1
WKV_BF16 = 0
WKV_MXFP8 = 1


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------
def decode_e4m3(codes) -> np.ndarray:
    """fp8 e4m3fn bit patterns -> float64, from the format's definition
    (OCP 8-bit floating point, E4M3: 1 sign bit, 4 exponent bits with bias 7,
    3 mantissa bits, subnormals at exponent 0, no infinities, NaN = S.1111.111).
    The table stores this type (``torch.float8_e4m3fn`` in the
    ``ParallelEngramEmbedding`` excerpt)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    sub = np.ldexp(m / 8.0, -6)
    mag = np.where(e == 0, sub, normal)
    out = sign * mag
    return np.where((e == 15) & ((c & 7) == 7), np.nan, out)


def decode_e8m0(codes) -> np.ndarray:
    """E8M0 scale bytes -> float64: 2^(code - 127), code 255 = NaN (OCP
    microscaling formats).  The pages' MXFP8 storage uses one per 32 channels
    (monishver11.github.io "DeepSeek's Other Modules", section "V4.1's two
    tables, reconciled")."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    out = np.ldexp(1.0, c - 127)
    return np.where(c == 255, np.nan, out)


def round_to_bf16(x) -> np.ndarray:
    """Round float values to bf16, nearest-even, returning uint16 bit patterns.

    bf16 keeps 8 significant bits and fp32's exponent range.  For finite x the
    result is the multiple of the quantum q = 2^(floor(log2|x|) - 7) (never
    below the subnormal quantum 2^-133) nearest to x, ties to the even
    multiple; np.rint rounds half to even and the scaling by a power of two is
    exact.  Values past the largest finite bf16 become infinities.  The value
    is rounded once, straight from float64."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    finite = np.isfinite(x)
    xf = np.where(finite, x, 0.0)
    _, e = np.frexp(xf)                       # xf = f * 2^e, 0.5 <= |f| < 1
    qexp = np.maximum(e - 8, -133)            # quantum exponent
    r = np.ldexp(np.rint(np.ldexp(xf, -qexp)), qexp)
    BF16_MAX = float.fromhex("0x1.fep127")
    r = np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, r), r)
    out[...] = np.where(finite, r, x)
    bits = out.astype(np.float32).view(np.uint32)   # exact: r is representable
    bits = (bits >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        bits = np.where(nan, np.uint16(0x7FC0), bits)
    return bits


def bf16_value(bits) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact widening)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# a1-a3: id range check, row gather, dequantisation
# --------------------------------------------------------------------------
def dequant_rows(codes, scales, scale_block: int, scale_fmt: int = SCALE_F32) -> np.ndarray:
    """Dequantise table rows to bf16 bits, as ``ParallelEngramEmbedding.forward``
    does: widen the codes to fp32, split each row into blocks of
    ``scale_block`` channels, multiply by the block's scale in fp32 (one
    rounding), cast to bf16.

    codes: uint8 [n, head_dim]; scales: [n, head_dim/scale_block] fp32, or uint8
    E8M0 codes when scale_fmt == SCALE_E8M0."""
    codes = np.asarray(codes, dtype=np.uint8)
    n, hd = codes.shape
    nb = hd // scale_block
    v = decode_e4m3(codes).astype(np.float32)           # exact
    if scale_fmt == SCALE_F32:
        s = np.asarray(scales, dtype=np.float32)
    else:
        s = decode_e8m0(scales).astype(np.float32)       # exact
    s = s.reshape(n, nb)
    prod = v.reshape(n, nb, scale_block) * s[:, :, None]  # float32 * float32 -> float32, RN
    return round_to_bf16(prod.reshape(n, hd).astype(np.float64))


def lookup(hash_ids, table, scale, scale_block: int, scale_fmt: int = SCALE_F32) -> np.ndarray:
    """Rows for each (token, column), flattened: bf16 bits [M, n_cols*head_dim]
    with element (m, c*head_dim + f) = dequantised row hash_ids[m, c], channel f
    (``Engram.forward``: ``self.embed(hash_ids).flatten(-2)``).

    An id outside [0, R) gives a row of +0.0: the sharded embedding maps such
    ids to local row 0 and then zeroes the row, and with one rank every id
    outside the table is outside the shard."""
    ids = np.asarray(hash_ids, dtype=np.int64)
    M, C = ids.shape
    table = np.asarray(table, dtype=np.uint8)
    R, hd = table.shape
    out = np.zeros((M, C, hd), dtype=np.uint16)
    valid = (ids >= 0) & (ids < R)
    if valid.any():
        r = ids[valid]
        out[valid] = dequant_rows(table[r], np.asarray(scale)[r], scale_block, scale_fmt)
    return out.reshape(M, C * hd)


def shard_bounds(num_rows: int, rank: int, world_size: int):
    """Rows [start, end) of the table held by `rank` when the table is split
    by rows over `world_size` ranks, as ``ParallelEngramEmbedding.__init__``
    splits it: part = ceil(num_rows / world_size) rows per rank, rank r from
    r*part.  The excerpt's last part may run past the table (its parameter is
    padded to `part` rows); here it ends at num_rows, since no id of the table
    reaches past it (an id >= num_rows gives a zero row, as with one rank)."""
    part = (num_rows + world_size - 1) // world_size
    start = rank * part
    return min(start, num_rows), min(start + part, num_rows)


def lookup_shard(hash_ids, table_shard, scale_shard, row_start: int, scale_block: int,
                 scale_fmt: int = SCALE_F32) -> np.ndarray:
    """One rank's rows before the exchange, as ``ParallelEngramEmbedding.forward``
    forms them: ids outside [row_start, row_start + shard rows) are masked,
    every id is made local (id - row_start, masked ones set to 0), the local
    row is looked up and dequantised, and masked rows are set to zero.
    Returns bf16 bits [M, n_cols*head_dim]."""
    ids = np.asarray(hash_ids, dtype=np.int64)
    M, C = ids.shape
    table_shard = np.asarray(table_shard, dtype=np.uint8)
    rows, hd = table_shard.shape
    mask = (ids < row_start) | (ids >= row_start + rows)
    local = np.where(mask, 0, ids - row_start)
    out = np.zeros((M, C, hd), dtype=np.uint16)
    if rows > 0:
        vals = dequant_rows(table_shard[local.reshape(-1)], np.asarray(scale_shard)[local.reshape(-1)], scale_block,
                            scale_fmt).reshape(M, C, hd)
        out = np.where(mask[:, :, None], np.uint16(0), vals)
    return out.reshape(M, C * hd)


# --------------------------------------------------------------------------
# a4: projection
# --------------------------------------------------------------------------
def project(e_bits, wkv_bits) -> np.ndarray:
    """kv = wkv(e): kv[m, j] = bf16( sum_k e[m, k] * W[j, k] ), W stored as the
    ``Linear``'s [out, in] weight (``Engram.__init__``: ``Linear(n_hash_cols *
    head_dim, dim * (hc_mult + 1))``).  The sum is taken in float64 (a library
    matrix product; bf16 x bf16 products are exact there) and rounded once."""
    e = bf16_value(e_bits)
    w = bf16_value(wkv_bits)
    return round_to_bf16(e @ w.T)


def mxfp8_weight(codes, scales, block: int = 32) -> np.ndarray:
    """The projection weight in the V4.1 FP8 format -> float64 [N, K], exact:
    W[j, k] = e4m3(codes[j, k]) * 2^(scales[j, k // block] - 127).

    monishver11.github.io "DeepSeek's Other Modules", section "V4.1's two
    tables, reconciled", says the tables and the projections are FP8, and
    zhuai.tech "Engram in DeepSeek V4.1 Flash" (section "Step 2: Read selected
    rows ...") describes the tables' MXFP8 format: E4M3 codes with one E8M0
    scale per 32 values.  The reading taken for the weight is the same format
    along its input dimension K (one scale per 32 consecutive inputs of an
    output row).  codes: uint8 [N, K]; scales: uint8 [N, K/block]."""
    c = np.asarray(codes, dtype=np.uint8)
    N, K = c.shape
    s = decode_e8m0(np.asarray(scales, dtype=np.uint8).reshape(N, K // block))
    return (decode_e4m3(c).reshape(N, K // block, block) * s[:, :, None]).reshape(N, K)


def project_mxfp8(e_bits, w_codes, w_scales, block: int = 32) -> np.ndarray:
    """kv = wkv(e) with the FP8 weight: kv[m, j] = bf16( sum_k e[m, k] * W[j, k] ),
    W = mxfp8_weight(w_codes, w_scales).  Products of a bf16 value and a
    block-scaled e4m3 value are exact in float64; the sum is taken in float64
    (a library matrix product) and rounded once."""
    e = bf16_value(e_bits)
    return round_to_bf16(e @ mxfp8_weight(w_codes, w_scales, block).T)


# --------------------------------------------------------------------------
# a5-a7: split, gate reductions, gate
# --------------------------------------------------------------------------
def gates(kv_bits, x_bits, q_bits, k_bits, mask=None, eps: float = 1e-6,
          clamp: float = 1e-6) -> np.ndarray:
    """Per (token, stream) gate, float64 [M, hc_mult], following
    ``Engram.forward``:

      key   = kv[:, :hc*dim] viewed [M, hc, dim] (stream-major);
      w     = q_weight * k_weight                     (elementwise, [hc, dim])
      rstd  = 1/sqrt(mean_d h^2 + eps) * 1/sqrt(mean_d key^2 + eps)
              -- per (token, stream), not jointly over the streams
      dot   = (sum_d h * w * key) * rstd * dim^-0.5
      gate  = sigmoid(copysign(sqrt(max(|dot|, clamp)), dot))
      gate  = 0 where the token mask is False."""
    x = bf16_value(x_bits)
    M, S, D = x.shape
    kv = bf16_value(kv_bits).reshape(M, -1)
    key = kv[:, :S * D].reshape(M, S, D)
    w = bf16_value(q_bits).reshape(S, D) * bf16_value(k_bits).reshape(S, D)
    mean_h2 = np.mean(x * x, axis=-1)
    mean_k2 = np.mean(key * key, axis=-1)
    rstd = (1.0 / np.sqrt(mean_h2 + eps)) * (1.0 / np.sqrt(mean_k2 + eps))
    dot = np.sum(x * w[None] * key, axis=-1) * rstd * (float(D) ** -0.5)
    z = np.copysign(np.sqrt(np.maximum(np.abs(dot), clamp)), dot)
    g = 1.0 / (1.0 + np.exp(-z))
    if mask is not None:
        g = np.where(np.asarray(mask).reshape(M, 1).astype(bool), g, 0.0)
    return g


# --------------------------------------------------------------------------
# a8: residual add
# --------------------------------------------------------------------------
def residual(kv_bits, x_bits, g, mask=None) -> np.ndarray:
    """out[m, s, d] = bf16( h[m, s, d] + g[m, s] * value[m, d] ), value =
    kv[:, hc*dim:] shared by the streams (``Engram.forward``'s last line);
    masked tokens return x's bits unchanged."""
    xb = np.asarray(x_bits, dtype=np.uint16)
    M, S, D = xb.shape
    x = bf16_value(xb)
    v = bf16_value(kv_bits).reshape(M, -1)[:, S * D:(S + 1) * D]
    with np.errstate(invalid="ignore", over="ignore"):   # masked rows are replaced below
        out = round_to_bf16(x + np.asarray(g, dtype=np.float64)[:, :, None] * v[:, None, :])
    if mask is not None:
        keep = ~np.asarray(mask).reshape(M).astype(bool)
        out[keep] = xb[keep]
    return out


# --------------------------------------------------------------------------
# the whole layer
# --------------------------------------------------------------------------
def forward(hash_ids, x_bits, table, scale, wkv_bits, q_bits, k_bits, mask=None,
            scale_block: int = 128, scale_fmt: int = SCALE_F32, eps: float = 1e-6,
            clamp: float = 1e-6, wkv_scale=None):
    """Engram layer: returns (out bf16 bits [M, hc, dim], gates float64 [M, hc],
    kv bf16 bits [M, dim*(hc+1)]).

    hash_ids: int64 [M, n_cols]; x_bits: uint16 [M, hc, dim]; table: uint8
    [R, head_dim]; scale: [R, head_dim/scale_block]; wkv_bits: uint16
    [dim*(hc+1), n_cols*head_dim]; q_bits, k_bits: uint16 [hc, dim]; mask:
    [M] truthy = apply, or None.  With wkv_scale given, wkv_bits holds the
    weight's e4m3 codes (uint8, same shape) and wkv_scale its E8M0 scales
    [dim*(hc+1), n_cols*head_dim/32] (project_mxfp8)."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    M = x_bits.shape[0]
    ids = np.asarray(hash_ids, dtype=np.int64).reshape(M, -1)
    e = lookup(ids, table, scale, scale_block, scale_fmt)
    kv = project(e, wkv_bits) if wkv_scale is None else project_mxfp8(e, wkv_bits, wkv_scale)
    g = gates(kv, x_bits, q_bits, k_bits, mask, eps, clamp)
    out = residual(kv, x_bits, g, mask)
    return out, g, kv


def parameter_count(num_rows: int, head_dim: int, n_cols: int, dim: int, hc_mult: int) -> int:
    """Learned parameters of one Engram instance, from the shapes the layer
    allocates: table [R, head_dim] + wkv [dim*(hc+1), n_cols*head_dim] +
    q_weight and k_weight [hc, dim] each (atlas.klimoza.dev "deepseek-v4.1 /
    engram-second", "Parameters" table; scales are not counted there)."""
    return num_rows * head_dim + (n_cols * head_dim) * (dim * (hc_mult + 1)) + 2 * hc_mult * dim
