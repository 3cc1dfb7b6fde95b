"""Seeded synthetic inputs for the Engram layer (host side).

This module is the only code shared by the CUDA path's harness and the CPU
oracle's harness.  It generates *inputs* and holds none of the layer's own
arithmetic: no fp8 decoding, no dequantisation, no projection, no gate.
Conversions of generated float values to bf16 / fp8 codes go through torch's
dtype casts (library routines), not through code of ours.

Randomness comes from two sources:

* numpy's PCG64 ``Generator`` for the small, host-made tensors (hash ids,
  hidden states, masks, ``wkv``, ``q_weight`` / ``k_weight``); they are made
  here and uploaded.
* a counter-based splitmix64 stream for the table (codes and scales), because
  the full-size table (384,016,682 rows x 256 B, about 98 GB) is filled on the
  device.  The device twin lives in ``csrc/synth.cu``; both implement the
  generator from its published definition (Steele, Lea & Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014, with the output
  mix constants of Vigna's public-domain ``splitmix64.c``):

      z   = key + (counter + 1) * 0x9E3779B97F4A7C15        (mod 2^64)
      z   = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
      z   = (z ^ (z >> 27)) * 0x94D049BB133111EB
      out = z ^ (z >> 31)

  Row ``r`` of the code table takes ``head_dim/4`` 64-bit draws (counter
  ``r*head_dim/4 + j``); each draw gives four 16-bit fields (low to high) that
  index a 65,536-entry quantile table of N(0,1) rounded to e4m3 codes.  Row
  ``r``'s scale block ``b`` takes counter ``r*nb + b`` of a second key; the top
  16 bits index a 65,536-entry fp32 quantile table of lognormal(0, 0.5).  The
  two quantile tables are built here once and handed to the device filler as
  inputs, so the device needs no transcendental function and both sides make
  byte-identical tables.

Workloads follow the five configurations of the layer's benchmark (tiny,
decode batch, Zipf prefill, skewed large decode, full-size table); their row
ranges are 24 consecutive primes above a base, as the V4.1 config's
``engram_num_embeddings`` are (atlas.klimoza.dev "deepseek-v4.1 / engram-second",
config.json; monishver11.github.io "DeepSeek's Other Modules", section
"V4.1's two tables, reconciled").
"""
from __future__ import annotations

import math
import statistics
from dataclasses import dataclass, field

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB

TAG_CODES = 1
TAG_SCALES = 2
TAG_WKV_CODES = 3
TAG_WKV_SCALES = 4


# --------------------------------------------------------------------------
# splitmix64, counter form
# --------------------------------------------------------------------------
def mix64(z: np.ndarray) -> np.ndarray:
    """splitmix64 output function on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX2)
    return z ^ (z >> np.uint64(31))


def mix64_int(z: int) -> int:
    """Scalar splitmix64 output function on a Python int."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tag: int) -> int:
    """Key of one named splitmix64 stream: mix64(seed * GAMMA + tag)."""
    return mix64_int((seed * GAMMA + tag) & MASK64)


def draw64(key: int, counters: np.ndarray) -> np.ndarray:
    """The counter-th output of the splitmix64 stream seeded with ``key``."""
    c = np.asarray(counters, dtype=np.uint64)
    z = np.uint64(key) + (c + np.uint64(1)) * np.uint64(GAMMA)
    return mix64(z)


# --------------------------------------------------------------------------
# row-range layout: consecutive primes
# --------------------------------------------------------------------------
def _is_prime(n: int) -> bool:
    if n < 2:
        return False
    if n % 2 == 0:
        return n == 2
    i = 3
    while i * i <= n:
        if n % i == 0:
            return False
        i += 2
    return True


def consecutive_primes_above(base: int, count: int, skip: int = 0) -> list[int]:
    """The primes strictly above ``base``, in ascending order, dropping the first ``skip``."""
    out: list[int] = []
    n = base
    while len(out) < count + skip:
        n += 1
        if _is_prime(n):
            out.append(n)
    return out[skip:]


def row_layout(prime_base: int, prime_skip: int, n_cols: int = 24):
    """(lengths, offsets) of the ``n_cols`` prime row ranges, column c owning
    rows [offsets[c], offsets[c] + lengths[c])."""
    lengths = np.array(consecutive_primes_above(prime_base, n_cols, prime_skip), dtype=np.int64)
    offsets = np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64)
    return lengths, offsets


# --------------------------------------------------------------------------
# quantile tables (built once; the device filler receives them as inputs)
# --------------------------------------------------------------------------
_QT_CACHE: dict = {}


def _normal_quantiles() -> np.ndarray:
    nd = statistics.NormalDist()
    return np.array([nd.inv_cdf((u + 0.5) / 65536.0) for u in range(65536)], dtype=np.float64)


def code_quantile_table() -> np.ndarray:
    """uint8[65536]: e4m3fn code of the N(0,1) quantile at (u+0.5)/65536,
    clipped to +-448 and cast by torch (round to nearest even)."""
    if "codes" not in _QT_CACHE:
        import torch
        q = np.clip(_normal_quantiles(), -448.0, 448.0).astype(np.float32)
        codes = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
        _QT_CACHE["codes"] = codes
    return _QT_CACHE["codes"]


def scale_quantile_table() -> np.ndarray:
    """float32[65536]: lognormal(0, 0.5) quantile at (u+0.5)/65536."""
    if "scales" not in _QT_CACHE:
        q = _normal_quantiles()
        _QT_CACHE["scales"] = np.array([math.exp(0.5 * v) for v in q], dtype=np.float32)
    return _QT_CACHE["scales"]


def e8m0_quantile_table() -> np.ndarray:
    """uint8[65536]: E8M0 code of the power of two nearest (in log2) to the
    lognormal(0, 0.5) quantile at (u+0.5)/65536: 127 + round(log2 q)."""
    if "e8m0" not in _QT_CACHE:
        q = scale_quantile_table().astype(np.float64)
        _QT_CACHE["e8m0"] = np.clip(127 + np.rint(np.log2(q)), 1, 254).astype(np.uint8)
    return _QT_CACHE["e8m0"]


# --------------------------------------------------------------------------
# table rows (host twin of the device filler)
# --------------------------------------------------------------------------
def table_rows(seed: int, rows: np.ndarray, head_dim: int = 256, scale_block: int = 128, scale_fmt: int = 0):
    """Codes (uint8 [n, head_dim]) and scales ([n, head_dim/scale_block]: fp32,
    or E8M0 bytes when scale_fmt == 1, drawn at the same stream positions) of
    the given table rows, exactly as the device filler writes them."""
    rows = np.asarray(rows, dtype=np.int64).reshape(-1)
    assert head_dim % 4 == 0 and head_dim % scale_block == 0
    words = head_dim // 4
    nb = head_dim // scale_block
    ctab = code_quantile_table()
    stab = scale_quantile_table()
    kc = stream_key(seed, TAG_CODES)
    ks = stream_key(seed, TAG_SCALES)
    cnt = rows.astype(np.uint64)[:, None] * np.uint64(words) + np.arange(words, dtype=np.uint64)[None, :]
    d = draw64(kc, cnt)                                            # [n, words]
    fields = np.stack([(d >> np.uint64(16 * q)) & np.uint64(0xFFFF) for q in range(4)], axis=-1)
    codes = ctab[fields.astype(np.int64)].reshape(rows.size, head_dim)
    scnt = rows.astype(np.uint64)[:, None] * np.uint64(nb) + np.arange(nb, dtype=np.uint64)[None, :]
    sidx = (draw64(ks, scnt) >> np.uint64(48)).astype(np.int64)
    if scale_fmt == 1:
        return codes.astype(np.uint8), e8m0_quantile_table()[sidx]
    scales = stab[sidx].astype(np.float32)
    return codes.astype(np.uint8), scales


def host_table(seed: int, num_rows: int, head_dim: int = 256, scale_block: int = 128, chunk: int = 1 << 16,
               scale_fmt: int = 0):
    """The whole table on the host (small tables only)."""
    codes = np.empty((num_rows, head_dim), dtype=np.uint8)
    scales = np.empty((num_rows, head_dim // scale_block), dtype=np.uint8 if scale_fmt == 1 else np.float32)
    for s in range(0, num_rows, chunk):
        e = min(num_rows, s + chunk)
        c, sc = table_rows(seed, np.arange(s, e), head_dim, scale_block, scale_fmt)
        codes[s:e] = c
        scales[s:e] = sc
    return codes, scales


# --------------------------------------------------------------------------
# bf16 helpers (library casts)
# --------------------------------------------------------------------------
def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float array -> uint16 bf16 bit patterns via torch's cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    prime_base: int
    prime_skip: int = 0
    ids: str = "uniform"          # uniform | zipf | hotset
    x_std: float = 1.0
    x_tiny_frac: float = 0.0      # fraction of (token, stream) vectors scaled by 1e-4
    mask: str = "all"             # all | span10 | frac5
    seed: int = 0
    dim: int = 5120
    hc_mult: int = 4
    n_cols: int = 24
    head_dim: int = 256
    scale_block: int = 128
    eps: float = 1e-6
    zipf_s: float = 1.1
    hot_rows: int = 1024
    fmt: str = "bf16"             # bf16: fp32 scales + bf16 wkv | mxfp8: E8M0/32 scales + FP8 wkv

    @property
    def scale_fmt(self) -> int:
        return 1 if self.fmt == "mxfp8" else 0

    @property
    def wkv_fmt(self) -> int:
        return 1 if self.fmt == "mxfp8" else 0

    @property
    def M(self) -> int:
        return self.B * self.T

    @property
    def K(self) -> int:
        return self.n_cols * self.head_dim

    @property
    def N(self) -> int:
        return self.dim * (self.hc_mult + 1)

    def layout(self):
        return row_layout(self.prime_base, self.prime_skip, self.n_cols)

    def num_rows(self) -> int:
        return int(self.layout()[0].sum())


WORKLOADS = [
    Workload("tiny_1x16", 1, 16, 4096, seed=0),
    Workload("decode_64x1", 64, 1, 1 << 20, seed=1),
    Workload("prefill_1x4096_zipf", 1, 4096, 1 << 24, ids="zipf", mask="span10", seed=2),
    Workload("decode_512x1_skew", 512, 1, 1 << 22, ids="hotset", x_std=math.sqrt(2.0),
             x_tiny_frac=0.01, seed=3),
    Workload("full_2x8192", 2, 8192, 16_000_000, prime_skip=24, mask="frac5", seed=4),
    # the V4.1-native formats: MXFP8 table (E8M0 per 32) and FP8 weight
    Workload("tiny_1x16_mxfp8", 1, 16, 4096, seed=5, scale_block=32, fmt="mxfp8"),
    Workload("decode_64x1_mxfp8", 64, 1, 1 << 20, seed=6, scale_block=32, fmt="mxfp8"),
    Workload("prefill_1x4096_mxfp8", 1, 4096, 1 << 22, mask="span10", seed=7, scale_block=32, fmt="mxfp8"),
]


def workload(name_or_index) -> Workload:
    if isinstance(name_or_index, int):
        return WORKLOADS[name_or_index]
    for w in WORKLOADS:
        if w.name == name_or_index:
            return w
    raise KeyError(name_or_index)


def make_hash_ids(w: Workload, lengths=None, offsets=None, rng=None) -> np.ndarray:
    """int64 [B, T, n_cols] global row ids, one per (token, column)."""
    if lengths is None:
        lengths, offsets = w.layout()
    rng = rng or np.random.default_rng([w.seed, 11])
    M = w.M
    out = np.empty((M, w.n_cols), dtype=np.int64)
    for c in range(w.n_cols):
        p = int(lengths[c])
        if w.ids == "uniform":
            local = rng.integers(0, p, size=M, dtype=np.int64)
        elif w.ids == "zipf":
            # truncated Zipf(s) over ranks 1..p by rejection, then a per-column
            # bijection rank -> row so hot ranks land on scattered rows
            rank = np.empty(M, dtype=np.int64)
            fill = 0
            while fill < M:
                r = rng.zipf(w.zipf_s, size=2 * (M - fill) + 16)
                r = r[(r >= 1) & (r <= p)]
                take = min(M - fill, r.size)
                rank[fill:fill + take] = r[:take]
                fill += take
            a = int(rng.integers(1, p))
            b = int(rng.integers(0, p))
            assert p < (1 << 31)  # (rank-1)*a + b stays below 2^62
            local = ((rank - 1) * a + b) % p
        elif w.ids == "hotset":
            hot = rng.choice(p, size=min(w.hot_rows, p), replace=False).astype(np.int64)
            is_hot = rng.random(M) < 0.5
            local = np.where(is_hot, hot[rng.integers(0, hot.size, size=M)],
                             rng.integers(0, p, size=M, dtype=np.int64))
        else:
            raise ValueError(w.ids)
        out[:, c] = local + offsets[c]
    return out.reshape(w.B, w.T, w.n_cols)


def make_x(w: Workload, rng=None, tokens: slice | None = None) -> np.ndarray:
    """bf16 bits [B, T, hc_mult, dim]."""
    rng = rng or np.random.default_rng([w.seed, 12])
    x = rng.standard_normal((w.M, w.hc_mult, w.dim), dtype=np.float32) * np.float32(w.x_std)
    if w.x_tiny_frac > 0:
        tiny = rng.random((w.M, w.hc_mult)) < w.x_tiny_frac
        x[tiny] *= np.float32(1e-4)
    return to_bf16_bits(x).reshape(w.B, w.T, w.hc_mult, w.dim)


def make_mask(w: Workload, rng=None) -> np.ndarray | None:
    """uint8 [B, T] (1 = Engram applies) or None when every entry is True."""
    rng = rng or np.random.default_rng([w.seed, 13])
    M = w.M
    if w.mask == "all":
        return None
    m = np.ones(M, dtype=np.uint8)
    if w.mask == "span10":
        span = int(round(0.10 * M))
        start = int(rng.integers(0, M - span + 1))
        m[start:start + span] = 0
    elif w.mask == "frac5":
        n_off = int(round(0.05 * M))
        m[rng.choice(M, size=n_off, replace=False)] = 0
    else:
        raise ValueError(w.mask)
    return m.reshape(w.B, w.T)


def make_wkv(w: Workload, rng=None) -> np.ndarray:
    """bf16 bits [N, K] = [dim*(hc_mult+1), n_cols*head_dim], entries N(0, 1/K)."""
    rng = rng or np.random.default_rng([w.seed, 14])
    a = rng.standard_normal((w.N, w.K), dtype=np.float32) * np.float32(1.0 / math.sqrt(w.K))
    return to_bf16_bits(a)


def make_wkv_mxfp8(w: Workload, rows_per_chunk: int = 1024):
    """FP8 weight: (e4m3 codes uint8 [N, K], E8M0 scales uint8 [N, K/32]).
    Codes are N(0,1) quantiles (the table's code quantile table) drawn from a
    counter stream, 4 codes per draw like the table; each 32-input block gets
    the scale 2^-7 or 2^-6 from the top bit of a second stream, so that the
    entries have about the bf16 weight's spread, N(0, 1/K)."""
    N, K = w.N, w.K
    assert K % 32 == 0
    ctab = code_quantile_table()
    kc = stream_key(w.seed, TAG_WKV_CODES)
    ks = stream_key(w.seed, TAG_WKV_SCALES)
    words = K // 4
    codes = np.empty((N, K), dtype=np.uint8)
    for j0 in range(0, N, rows_per_chunk):
        j1 = min(N, j0 + rows_per_chunk)
        cnt = np.arange(j0, j1, dtype=np.uint64)[:, None] * np.uint64(words) + np.arange(words, dtype=np.uint64)[None, :]
        d = draw64(kc, cnt)
        f = np.stack([(d >> np.uint64(16 * q)) & np.uint64(0xFFFF) for q in range(4)], axis=-1)
        codes[j0:j1] = ctab[f.astype(np.int64)].reshape(j1 - j0, K)
    nb = K // 32
    top = draw64(ks, np.arange(N * nb, dtype=np.uint64)) >> np.uint64(63)
    scales = (np.uint64(120) + top).astype(np.uint8).reshape(N, nb)
    return codes, scales


def make_qk(w: Workload, rng=None):
    """bf16 bits q_weight, k_weight [hc_mult, dim], entries 1 + N(0, 0.1)."""
    rng = rng or np.random.default_rng([w.seed, 15])
    sd = np.float32(math.sqrt(0.1))
    q = 1.0 + rng.standard_normal((w.hc_mult, w.dim), dtype=np.float32) * sd
    k = 1.0 + rng.standard_normal((w.hc_mult, w.dim), dtype=np.float32) * sd
    return to_bf16_bits(q), to_bf16_bits(k)


@dataclass
class HostInputs:
    """Everything but the table, on the host."""
    w: Workload
    hash_ids: np.ndarray
    x: np.ndarray
    mask: np.ndarray | None
    wkv: np.ndarray               # bf16 bits, or e4m3 codes for the mxfp8 format
    q: np.ndarray
    k: np.ndarray
    lengths: np.ndarray = field(default=None)
    offsets: np.ndarray = field(default=None)
    wkv_scale: np.ndarray | None = None   # E8M0 [N, K/32] for the mxfp8 format


def make_inputs(w: Workload) -> HostInputs:
    lengths, offsets = w.layout()
    q, k = make_qk(w)
    wkv_scale = None
    if w.fmt == "mxfp8":
        wkv, wkv_scale = make_wkv_mxfp8(w)
    else:
        wkv = make_wkv(w)
    return HostInputs(w=w, hash_ids=make_hash_ids(w, lengths, offsets), x=make_x(w),
                      mask=make_mask(w), wkv=wkv, q=q, k=k,
                      lengths=lengths, offsets=offsets, wkv_scale=wkv_scale)
