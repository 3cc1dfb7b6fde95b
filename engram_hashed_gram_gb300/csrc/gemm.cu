// Step a4 of the Engram layer, the wkv projection (atlas.klimoza.dev
// "deepseek-v4.1 / engram-second", `Engram.forward`:
// kv = wkv(embed(hash_ids).flatten(-2))): kv[m, n] = sum_k E[m, k] * W[n, k],
// E the gathered bf16 rows [M, K], W the Linear's [N, K] bf16 weight, fp32
// accumulation.
//
// Design (sm_103a, one CTA per SM, persistent):
//  * a work unit is a 128 x 256 output tile over the whole K (decode: the 100
//    tiles on 100 CTAs already stream the weight at the HBM rate), or over
//    one K range (split-K for fewer tiles or a capped SM budget, or the
//    remainder split of a small last wave); units are dealt round-robin to
//    the CTAs;
//  * warp 0 (one thread) streams A = E[A_ROWS rows, 64 k] with a 2-D TMA copy
//    (128-byte swizzle) and B = W[256 rows, 64 k] as one contiguous 32 KB bulk
//    copy of the weight's tile-packed copy (packed at create time exactly as
//    the swizzled copy would land) into a STAGES-deep shared-memory ring; the
//    first stages' B copies go out before the wait for the gather;
//  * warp 1 (one thread) issues tcgen05.mma (M=128, N=256, K=16, bf16 -> fp32)
//    into one of two 256-column tensor-memory accumulators and commits each
//    stage back to the producer;
//  * warps 2-5 drain the other accumulator with tcgen05.ld and write either the
//    bf16 kv (round to nearest even) or the fp32 partial sums of a K range,
//    through a per-warp shared-memory tile so that stores are row segments;
//  * no cluster, no multicast: the L2 serves the reuse of E and W across CTAs.
// FP8 (the MXFP8 weight): A and B are e4m3 codes, K = 128 per stage, the E8M0
// scales ride with each stage and tcgen05.cp moves them into tensor memory
// for tcgen05.mma kind::mxf8f6f4.block_scale (one accumulator: the scales use
// the second one's columns).  BULK (bf16, 2,048 tokens and more): the
// epilogue sends each lane's row segment with a bulk copy.  FUSED: the gate
// and the residual add run in the epilogue (engram_config.fuse_gate).
// Variants: A_ROWS = 128 with 4 stages in general; for batches of at most 64
// or 32 tokens the A box holds only 64 or 32 rows, and the shared memory that
// frees goes to a deeper ring (5 stages), i.e. more of the weight stream in
// flight per SM.  The MMA still reads 128 rows of A: rows past the box are
// whatever the neighbouring shared memory holds, their accumulator rows are
// never stored, and a row of D depends on its own row of A only.  Rows of the
// last M tile past M read as zeros (TMA bounds fill) and are not stored.
//
// MXFP8 weight (FP8 = true): A is the gathered table codes (e4m3, [M, K]) and
// B the weight's codes, each with one E8M0 scale per 32 K per row; a stage is
// K = 128 (still 128 bytes per row), plus the stage's scales: 512 bytes for
// the 128 rows of A and 1 KB for the 256 rows of B, each a 32-line x 16-byte
// block in which line l holds the 4 scales (one per 32 K) of rows l, l+32,
// l+64, l+96.  The MMA thread copies them into tensor memory (tcgen05.cp,
// 32x128b replicated to the four lane quarters) and issues four
// tcgen05.mma.kind::mxf8f6f4.block_scale (K = 32 each; the instruction
// descriptor picks the scale byte).  The accumulator is single-buffered: the
// scales take tensor-memory columns 256 and up.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.cuh"

namespace engram {
namespace {

constexpr int kBBytes = kBN * kBK * 2;        // 32 KB
constexpr uint32_t kTmemCols = 2 * kBN;        // two fp32 accumulators (bf16), or one + scales (FP8)
constexpr int kKB8 = 128;                      // K elements per FP8 stage (128 bytes per row)
constexpr int kSfaBytes = 512;                 // scales of 128 A rows x 4 K-blocks of 32
constexpr int kSfbBytes = 1024;                // scales of 256 B rows x 4
constexpr uint32_t kSfCol0 = kBN;              // first tensor-memory column of the FP8 scales
constexpr uint32_t kSfColsPerStage = 16;       // A: 4 columns, B: 8 columns

constexpr int kMaxStreams = 4;                 // hc_mult
constexpr int kMaxBlocks = 5120 / kBN;         // 256-channel blocks per stream (dim <= 5120)

// Per epilogue warp, fused mode only: 32 rows x 32 bf16 of a value tile
// (pitch 80 bytes: conflict-free 16-byte accesses), the rows' gates and
// pass-through flags.  Key tiles use its first 1 KB for the tile's q*k.
constexpr int kEpiPitch = 80;
constexpr int kEpiGates = 32 * kEpiPitch;            // float [32][4]
constexpr int kEpiFlags = kEpiGates + 32 * 16;       // int [32]
constexpr int kEpiWarpBytes = kEpiFlags + 32 * 4;    // 3,200

// Fused mode: the units a CTA works on come from a global ticket counter (see
// the kernel), and its producer hands each one to the MMA thread and the four
// epilogue warps through a ring of kRing slots in shared memory: the unit
// index, a "full" barrier (producer -> consumers) and an "empty" barrier
// (5 consumer arrivals -> producer).
constexpr int kRing = 8;
constexpr int kRingBytes = kRing * 8 + 2 * kRing * 8;

// Per epilogue warp, plain mode: a 32-row x 32-column fp32 tile (pitch 144
// bytes, so that 16-byte writes of a row per lane and 16-byte reads of 8
// lanes along a row are both free of bank conflicts).
constexpr int kPlainPitch = 144;
constexpr int kPlainWarpBytes = 32 * kPlainPitch;    // 4,608

template <int A_ROWS, int STAGES, bool FP8 = false>
struct Cfg {
  static constexpr int kABytes = A_ROWS * kBK * 2;                  // A_ROWS x 128 bytes either way
  static constexpr int kSfBytes = FP8 ? kSfaBytes + kSfbBytes : 0;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfBytes;  // bytes one stage's copies deliver
  static constexpr int kSfOffset = STAGES * (kABytes + kBBytes);
  static constexpr int kBarOffset = STAGES * kStageBytes;
  static constexpr int kNumBars = 2 * STAGES + 2 + 2 + 1;
  static constexpr int kEpiOffset = kBarOffset + 256;              // epilogue staging, after the barriers
  static constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + kEpiOffset + 4 * kPlainWarpBytes;
  static constexpr size_t kRingOffset = kEpiOffset + 4 * kEpiWarpBytes;   // fused: the CTA's unit queue
  static constexpr size_t kSmemFused = 1024 + kRingOffset + kRingBytes;
  static constexpr bool kCanFuse = !FP8 && kSmemFused <= 232448;
  static_assert(!kCanFuse || kSmemFused <= 232448, "fused-mode shared memory");
  static_assert(!FP8 || STAGES * kSfColsPerStage + kSfCol0 <= kTmemCols, "scale columns");
  static_assert(kNumBars * 8 + 8 <= 256, "barrier area");
  static_assert(kABytes % 1024 == 0, "A stages must stay 1024-byte aligned");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

// Tile t of an m_tiles x n_count grid, rasterised in groups of group_m M tiles
// (M fastest inside a group) so that tiles running at the same time share
// their A and B tiles in L2.
__device__ __forceinline__ void raster(const GemmArgs& a, int64_t t, int n_count, int& mt, int& ntl) {
  const int64_t group_tiles = static_cast<int64_t>(a.group_m) * n_count;
  const int64_t g = t / group_tiles;
  const int64_t r = t - g * group_tiles;
  const int gm0 = static_cast<int>(g) * a.group_m;
  const int gm = min(a.group_m, a.m_tiles - gm0);
  ntl = static_cast<int>(r / gm);
  mt = gm0 + static_cast<int>(r % gm);
}

__device__ __forceinline__ bool remainder_unit(const GemmArgs& a, int64_t u) {
  return a.rem_splits > 0 && u >= a.full_units;
}

// Fused mode: unit u -> (M tile, N tile).  The M tiles are taken in groups of
// group_m; K(g) is the key tiles of group g, V(g) its value tiles, each
// rasterised with M fastest.  The order is
//     K(0), K(1), V(0), K(2), V(1), ..., K(G-1), V(G-2), V(G-1)
// so that a value tile, whose epilogue needs the gates of its rows and so all
// key tiles of its M tile, comes a whole group of key tiles after them (they
// are long finished by then), and the value tiles' heavier epilogues (x and
// out of every stream) are spread over the run instead of bunched at its end.
// Every unit a value tile waits for has a smaller index.  m_count is the
// number of M units: M tiles, or M pairs for the CTA-pair kernel.
__device__ __forceinline__ void fused_coords(const GemmArgs& a, int64_t u, int m_count, int& mt, int& nt) {
  const int KT = a.key_n_tiles;
  const int VT = a.n_tiles - a.key_n_tiles;
  const int G = (m_count + a.group_m - 1) / a.group_m;
  int64_t off = 0;
  for (int seg = 0; seg < 2 * G; ++seg) {
    int g;
    bool key;
    if (seg == 0) {
      g = 0, key = true;
    } else if (seg == 2 * G - 1) {
      g = G - 1, key = false;
    } else if (seg & 1) {
      g = (seg + 1) >> 1, key = true;
    } else {
      g = (seg >> 1) - 1, key = false;
    }
    const int gm = min(a.group_m, m_count - g * a.group_m);
    const int64_t size = static_cast<int64_t>(gm) * (key ? KT : VT);
    if (u < off + size) {
      const int64_t l = u - off;
      mt = g * a.group_m + static_cast<int>(l % gm);
      nt = static_cast<int>(l / gm) + (key ? 0 : KT);
      return;
    }
    off += size;
  }
  mt = 0, nt = 0;   // u >= units: not reached
}

template <bool FUSED>
__device__ __forceinline__ void unit_coords(const GemmArgs& a, int64_t u, int& mt, int& nt, int& sp) {
  if (!FUSED && remainder_unit(a, u)) {             // a remainder unit: sp is its K range
    const int64_t j = u - a.full_units;
    sp = static_cast<int>(j % a.rem_splits);
    const int64_t tiles = static_cast<int64_t>(a.m_tiles) * a.n_tiles;
    raster(a, tiles - a.rem_tiles + j / a.rem_splits, a.n_tiles, mt, nt);
    return;
  }
  sp = static_cast<int>(u % a.splits);
  const int64_t t = u / a.splits;
  if constexpr (FUSED) {
    fused_coords(a, t, a.m_tiles, mt, nt);
    return;
  }
  raster(a, t, a.n_tiles, mt, nt);
}

// K blocks of unit u: [first, first + count).
__device__ __forceinline__ void unit_kb(const GemmArgs& a, int64_t u, int sp, int& first, int& count) {
  if (remainder_unit(a, u)) {
    first = sp * a.rem_kb;
    count = a.rem_kb;
  } else {
    first = sp * a.kb_per_split;
    count = a.kb_per_split;
  }
}

// The weight tile (N tile nt, K block kb) into a B stage: one contiguous 32 KB
// copy from the packed weight, or a 2-D tensor copy of the row-major weight.
// FP8: the tile's scales (1 KB, packed the same way) go to the stage's B-scale
// block.  kbt = K blocks per row of tiles.
template <bool FP8>
__device__ __forceinline__ void load_b(const GemmArgs& a, const CUtensorMap& tmB, uint8_t* dst, uint8_t* sf_dst,
                                       uint64_t* bar, int nt, int kb, int kbt, uint64_t policy) {
  const int64_t tile = static_cast<int64_t>(nt) * kbt + kb;
  if constexpr (FP8) {
    bulk_load_hint(dst, a.wpack + tile * kBBytes, kBBytes, bar, policy);
    bulk_load_hint(sf_dst + kSfaBytes, a.sfb + tile * kSfbBytes, kSfbBytes, bar, policy);
  } else if (a.wpack != nullptr) {
    bulk_load_hint(dst, a.wpack + tile * kBBytes, kBBytes, bar, policy);
  } else {
    tma_load_2d_hint(dst, &tmB, bar, kb * kBK, nt * kBN, policy);
  }
}

// The gathered rows (M tile mt, K block kb) into an A stage; FP8: with their
// scales (512 bytes, from the gather) into the stage's A-scale block.
template <bool FP8>
__device__ __forceinline__ void load_a(const GemmArgs& a, const CUtensorMap& tmA, uint8_t* dst, uint8_t* sf_dst,
                                       uint64_t* bar, int mt, int kb, int kbt) {
  if constexpr (FP8) {
    tma_load_2d(dst, &tmA, bar, kb * kKB8, mt * kBM);
    bulk_load_hint(sf_dst, a.sfa + (static_cast<int64_t>(mt) * kbt + kb) * kSfaBytes, kSfaBytes, bar,
                   policy_evict_last());
  } else {
    tma_load_2d(dst, &tmA, bar, kb * kBK, mt * kBM);
  }
}

__device__ __forceinline__ void raise_abort(volatile int* abort_flag, unsigned long long* err) {
  *abort_flag = 1;
  atomicOr(err, kErrTimeout);
}

// kv (bf16) or the fp32 split-K partial sums of the warp's 32 rows (m0 ..
// m0+31), columns [nt*256, nt*256 + 256).  tcgen05.ld gives each lane one
// row; every 32-column chunk goes through the warp's shared-memory tile, and
// from there either
//  * (BULK, chosen by a.bulk_epilogue) each lane sends its row's chunk with one bulk copy
//    (128 bytes of fp32 or 64 of bf16) and never waits on the stores: before
//    its line is rewritten it waits only for the previous copy to have read
//    it, and for completion once, at the end of the unit.  Large bf16
//    batches use this; while the weight streams (decode), or with the MXFP8
//    operands' many small scale copies, the row copies would queue behind the
//    loads in the copy engine, so there
//  * the warp reads the tile back by row segments and stores them (8 lanes
//    write one row's 128 bytes of fp32, or 4 lanes its 64 bytes of bf16).
// tile / tile_stride: instead of the output, the fp32 sums go to this 32-row
// block (row r at tile + r * tile_stride), as for a remainder unit.
template <bool BULK>
__device__ __forceinline__ void plain_epilogue(const GemmArgs& a, uint32_t t_row, int64_t m0, int nt, int sp,
                                               int lane, uint32_t stage, float* tile = nullptr,
                                               int64_t tile_stride = 0) {
  if (m0 >= a.M) return;                             // no row of this quarter is a token
  const bool bf16 = tile == nullptr && a.out_mode == kOutBf16;
  const uint32_t mine = stage + static_cast<uint32_t>(lane * kPlainPitch);
  constexpr bool bulk = BULK;
  const bool mine_valid = m0 + lane < a.M;
  uint8_t* row_dst;                                  // bulk mode: this lane's row, first column of the tile
  if (tile != nullptr) {
    row_dst = reinterpret_cast<uint8_t*>(tile + lane * tile_stride);
  } else if (bf16) {
    row_dst = reinterpret_cast<uint8_t*>(a.kv + (m0 + lane) * a.N + nt * kBN);
  } else {
    row_dst = reinterpret_cast<uint8_t*>(a.part + (static_cast<int64_t>(sp) * a.M + m0 + lane) * a.N + nt * kBN);
  }
#pragma unroll 1
  for (int c = 0; c < kBN / 32; ++c) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), r);
    tmem_ld_wait();
    if constexpr (bulk) bulk_wait_read_all();        // the previous chunk's copy has left the line
    if (bf16) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        st_shared_v4(mine + 16 * j,
                     make_uint4(pack_bf16x2(__uint_as_float(r[8 * j + 0]), __uint_as_float(r[8 * j + 1])),
                                pack_bf16x2(__uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3])),
                                pack_bf16x2(__uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5])),
                                pack_bf16x2(__uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7]))));
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) st_shared_v4(mine + 16 * j, make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]));
    }
    if constexpr (bulk) {
      fence_proxy_async_shared();                    // the line is visible to the bulk copy
      if (mine_valid) {
        bulk_store(row_dst + (bf16 ? c * 64 : c * 128), mine, bf16 ? 64u : 128u);
        bulk_commit();
      }
      continue;
    }
    __syncwarp();
    const int n0 = nt * kBN + c * 32;
    if (bf16) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = i * 8 + (lane >> 2);
        const int q = lane & 3;
        if (m0 + row < a.M) {
          const uint4 v = ld_shared_v4(stage + static_cast<uint32_t>(row * kPlainPitch + q * 16));
          *reinterpret_cast<uint4*>(a.kv + (m0 + row) * a.N + n0 + q * 8) = v;
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int row = i * 4 + (lane >> 3);
        const int q = lane & 7;
        if (m0 + row < a.M) {
          const uint4 v = ld_shared_v4(stage + static_cast<uint32_t>(row * kPlainPitch + q * 16));
          float* dst = tile != nullptr ? tile + row * tile_stride + c * 32 + q * 4
                                       : a.part + (static_cast<int64_t>(sp) * a.M + m0 + row) * a.N + n0 + q * 4;
          *reinterpret_cast<uint4*>(dst) = v;
        }
      }
    }
    __syncwarp();                                    // the tile is rewritten by the next chunk
  }
  if constexpr (bulk) bulk_wait_all();               // the unit's rows are in global memory
}

// bf16 kv of the warp's 32 rows for the FP8 kernel, whose single accumulator
// keeps the next tile's MMAs waiting for the epilogue: the lane's whole row
// (256 columns, as 128 bf16 pairs in registers) leaves tensor memory first,
// the accumulator is released (tempty_bar), and only then does the row go out
// through the warp's shared-memory tile, as in plain_epilogue's bf16 path and
// with the same values.
__device__ __forceinline__ void bf16_epilogue_release_first(const GemmArgs& a, uint32_t t_row, int64_t m0, int nt,
                                                            int lane, uint32_t stage, uint64_t* tempty_bar) {
  const bool any = m0 < a.M;                         // some row of this quarter is a token
  uint32_t packed[kBN / 32][16];
  if (any) {
#pragma unroll
    for (int c = 0; c < kBN / 32; ++c) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) packed[c][j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
    }
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(tempty_bar);
  if (!any) return;
  const uint32_t mine = stage + static_cast<uint32_t>(lane * kPlainPitch);
#pragma unroll
  for (int c = 0; c < kBN / 32; ++c) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      st_shared_v4(mine + 16 * j,
                   make_uint4(packed[c][4 * j], packed[c][4 * j + 1], packed[c][4 * j + 2], packed[c][4 * j + 3]));
    __syncwarp();
    const int n0 = nt * kBN + c * 32;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = i * 8 + (lane >> 2);
      const int q = lane & 3;
      if (m0 + row < a.M) {
        const uint4 v = ld_shared_v4(stage + static_cast<uint32_t>(row * kPlainPitch + q * 16));
        *reinterpret_cast<uint4*>(a.kv + (m0 + row) * a.N + n0 + q * 8) = v;
      }
    }
    __syncwarp();                                    // the tile is rewritten by the next chunk
  }
}

// ---------------------------------------------------------------- fused epilogue
// The fused epilogue forms the gate kernel's sums in the gate kernel's order
// (gate.cu): a 256-channel block of one stream is 32 groups of 8 channels; a
// group's sum is an fmaf chain over its channels from 0; the 32 group sums
// combine as an xor butterfly over 32 lanes would (x_l + x_{l+16} for l < 16,
// then + x_{l+8} for l < 8, ... -- IEEE addition is commutative, so every lane
// of the butterfly holds these bits); blocks are added in block order from 0.
// With the same bf16 kv values (this kernel's accumulators rounded as
// lookup_project rounds them) the gates and outputs equal those of
// lookup_project followed by gate_apply, bit for bit.

__device__ __forceinline__ void unpack8_bf16(uint4 v, float* f) {
  f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xFFFF0000u);
  f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xFFFF0000u);
  f[4] = __uint_as_float(v.z << 16); f[5] = __uint_as_float(v.z & 0xFFFF0000u);
  f[6] = __uint_as_float(v.w << 16); f[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

// Key tile: row m's block sums of stream s, channels [d0, d0 + 256).  The warp
// first copies the tile's 256 weight products (the same for every row) to its
// shared memory; row m's hidden state is loaded one 32-channel chunk ahead.
__device__ __forceinline__ void fused_key_epilogue(const GemmArgs& a, uint32_t t_row, int64_t m, int n0, int lane,
                                                   float* wsm) {
  const int s = n0 / a.dim;
  const int d0 = n0 - s * a.dim;
  const bool active = m < a.M && (a.mask == nullptr || a.mask[m] != 0);
  const uint4* xr = reinterpret_cast<const uint4*>(a.x + (m * a.hc + s) * a.dim + d0);
  {
    const float4* wg = reinterpret_cast<const float4*>(a.wprod + static_cast<int64_t>(s) * a.dim + d0) + 2 * lane;
    reinterpret_cast<float4*>(wsm)[2 * lane] = __ldg(wg);
    reinterpret_cast<float4*>(wsm)[2 * lane + 1] = __ldg(wg + 1);
    __syncwarp();
  }
  float th[16], tk[16], td[16];   // the butterfly after its first step
  uint4 hcur[4], hnext[4];
  if (active) {
#pragma unroll
    for (int g = 0; g < 4; ++g) hcur[g] = __ldg(xr + g);
  }
#pragma unroll
  for (int c = 0; c < kBN / 32; ++c) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), r);
    if (active && c + 1 < kBN / 32) {
#pragma unroll
      for (int g = 0; g < 4; ++g) hnext[g] = __ldg(xr + 4 * (c + 1) + g);
    }
    tmem_ld_wait();
    if (active) {
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int l = 4 * c + g;                     // group index in the block
        float h[8];
        unpack8_bf16(hcur[g], h);
        const float4 w0 = reinterpret_cast<const float4*>(wsm)[2 * l];
        const float4 w1 = reinterpret_cast<const float4*>(wsm)[2 * l + 1];
        const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        float sh = 0.0f, sk = 0.0f, sd = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float k = round_bf16(__uint_as_float(r[8 * g + j]));
          sh = fmaf(h[j], h[j], sh);
          sk = fmaf(k, k, sk);
          sd = fmaf(__fmul_rn(h[j], w[j]), k, sd);
        }
        if (l < 16) {
          th[l] = sh; tk[l] = sk; td[l] = sd;
        } else {                                     // butterfly step 16
          th[l - 16] = th[l - 16] + sh; tk[l - 16] = tk[l - 16] + sk; td[l - 16] = td[l - 16] + sd;
        }
      }
#pragma unroll
      for (int g = 0; g < 4; ++g) hcur[g] = hnext[g];
    }
  }
  __syncwarp();                                      // wsm is rewritten by the next tile
  if (active) {
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) {
#pragma unroll
      for (int l = 0; l < off; ++l) {
        th[l] = th[l] + th[l + off]; tk[l] = tk[l] + tk[l + off]; td[l] = td[l] + td[l + off];
      }
    }
    const int nblk = a.dim / kBN;
    reinterpret_cast<float4*>(a.gsum)[(m * a.hc + s) * nblk + d0 / kBN] = make_float4(th[0], tk[0], td[0], 0.0f);
  }
}

// Called by every key-tile warp after its block sums are written.  The last
// warp to arrive for an (M tile, lane quarter) -- the counter's old value tells
// it -- forms the gates of the quarter's 32 rows from all block sums, stores
// them and raises the quarter's ready flag, so that value tiles read one float4
// per row instead of summing the blocks themselves.
__device__ __forceinline__ void fused_key_publish(const GemmArgs& a, int64_t m, int mt, int q, int lane) {
  __syncwarp();
  uint32_t old = 0;
  if (lane == 0) old = atom_acq_rel_add_u32(a.counters + mt * 8 + q, 1u);
  old = __shfl_sync(0xFFFFFFFFu, old, 0);
  if (old + 1 != static_cast<uint32_t>(a.key_n_tiles)) return;
  __threadfence();                                   // every block sum of these rows is visible now
  if (m < a.M) {
    float g[kMaxStreams] = {};
    if (a.mask == nullptr || a.mask[m] != 0) {
      const int nblk = a.dim / kBN;
#pragma unroll
      for (int s = 0; s < kMaxStreams; ++s) {
        if (s >= a.hc) break;
        const float4* p = reinterpret_cast<const float4*>(a.gsum) + (m * a.hc + s) * nblk;
        float sh = 0.0f, sk = 0.0f, sd = 0.0f;
#pragma unroll
        for (int b0 = 0; b0 < kMaxBlocks; b0 += kMaxBlocks / 2) {   // two batches of loads in flight
          float4 blk[kMaxBlocks / 2];
#pragma unroll
          for (int b = 0; b < kMaxBlocks / 2; ++b)
            if (b0 + b < nblk) blk[b] = __ldcg(p + b0 + b);
#pragma unroll
          for (int b = 0; b < kMaxBlocks / 2; ++b) {  // block order
            if (b0 + b < nblk) {
              sh += blk[b].x;
              sk += blk[b].y;
              sd += blk[b].z;
            }
          }
        }
        g[s] = engram_gate(sh, sk, sd, a.dim, a.eps, a.clamp, a.inv_sqrt_dim);
      }
    }
    reinterpret_cast<float4*>(a.gates)[m] = make_float4(g[0], g[1], g[2], g[3]);
  }
  __syncwarp();
  // (the test hook withholds the flag, so that the value tiles' bounded wait runs out)
  if (lane == 0 && !a.hold_ready_flags) red_release_add_u32(a.counters + mt * 8 + 4 + q, 1u);
}

// Value tile: once the gates of the warp's 32 rows are ready, out = h + gate *
// value for channels [d0, d0 + 256) of every stream.  Each 32-channel chunk of
// the value passes through the warp's shared-memory tile so that 4 lanes cover
// one row's 64 contiguous bytes of x and out (8 rows per warp instruction
// instead of 32).  Returns false if the wait ran out.
__device__ __forceinline__ bool fused_value_epilogue(const GemmArgs& a, uint32_t t_row, int64_t m, int mt, int q,
                                                     int n0, int lane, volatile int* abort_flag, uint8_t* epi) {
  const int d0 = n0 - a.hc * a.dim;
  bool ok = true;
  if (lane == 0) {
    const unsigned long long t0 = globaltimer_ns();
    while (ld_acquire_u32(a.counters + mt * 8 + 4 + q) == 0u) {
      if (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) {
        ok = false;
        break;
      }
      __nanosleep(64);
    }
  }
  ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
  if (!ok) return false;
  __threadfence();
  float* gsm = reinterpret_cast<float*>(epi + kEpiGates);
  int* fsm = reinterpret_cast<int*>(epi + kEpiFlags);
  {
    const bool active = m < a.M;
    const bool pass = active && a.mask != nullptr && a.mask[m] == 0;
    reinterpret_cast<float4*>(gsm)[lane] =
        active && !pass ? __ldcg(reinterpret_cast<const float4*>(a.gates) + m) : make_float4(0.f, 0.f, 0.f, 0.f);
    fsm[lane] = active ? (pass ? 2 : 1) : 0;
  }
  __syncwarp();
  const int64_t m0 = m - lane;                       // the warp's first row
  const int cg = (lane & 3) * 8;                     // this lane's 8 channels of a chunk
  int flag[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) flag[i] = fsm[(lane >> 2) + 8 * i];
#pragma unroll 1
  for (int c = 0; c < kBN / 32; ++c) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), r);
    tmem_ld_wait();
    uint4* vrow = reinterpret_cast<uint4*>(epi + lane * kEpiPitch);
#pragma unroll
    for (int j = 0; j < 4; ++j)                      // kv rounded to bf16, as the projection returns it
      vrow[j] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * j + 0]), __uint_as_float(r[8 * j + 1])),
                           pack_bf16x2(__uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3])),
                           pack_bf16x2(__uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5])),
                           pack_bf16x2(__uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7])));
    __syncwarp();
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint4 hb[2][kMaxStreams];                      // half of the chunk's x loads in flight together
#pragma unroll
      for (int ii = 0; ii < 2; ++ii) {
        const int i = 2 * half + ii;
        const uint4* xr =
            reinterpret_cast<const uint4*>(a.x + ((m0 + (lane >> 2) + 8 * i) * a.hc) * a.dim + d0 + c * 32 + cg);
#pragma unroll
        for (int s = 0; s < kMaxStreams; ++s)
          if (flag[i] != 0 && s < a.hc) hb[ii][s] = __ldg(xr + s * (a.dim / 8));
      }
#pragma unroll
      for (int ii = 0; ii < 2; ++ii) {
        const int i = 2 * half + ii;
        if (flag[i] == 0) continue;
        const int rl = (lane >> 2) + 8 * i;
        const int64_t mr = m0 + rl;
        float v[8];
        unpack8_bf16(*reinterpret_cast<const uint4*>(epi + rl * kEpiPitch + cg * 2), v);
#pragma unroll
        for (int s = 0; s < kMaxStreams; ++s) {
          if (s >= a.hc) break;
          uint4 o = hb[ii][s];
          if (flag[i] == 1) {
            const float gs = gsm[4 * rl + s];
            float h[8];
            unpack8_bf16(hb[ii][s], h);
            o.x = pack_bf16x2(fmaf(gs, v[0], h[0]), fmaf(gs, v[1], h[1]));
            o.y = pack_bf16x2(fmaf(gs, v[2], h[2]), fmaf(gs, v[3], h[3]));
            o.z = pack_bf16x2(fmaf(gs, v[4], h[4]), fmaf(gs, v[5], h[5]));
            o.w = pack_bf16x2(fmaf(gs, v[6], h[6]), fmaf(gs, v[7], h[7]));
          }
          *reinterpret_cast<uint4*>(a.out + (mr * a.hc + s) * a.dim + d0 + c * 32 + cg) = o;
        }
      }
    }
    __syncwarp();                                    // the tile is rewritten by the next chunk
  }
  return true;
}

// FUSED selects the gate epilogue at compile time, so that the plain kernel
// carries none of its registers; FP8 the block-scaled MXFP8 operands.
template <int A_ROWS, int STAGES, bool FUSED, bool FP8, bool BULK = false>
__global__ void __launch_bounds__(kGemmThreads, 1)
    wkv_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmArgs a) {
  static_assert(!(FUSED && FP8), "the fused epilogue takes bf16 weights only");
  using C = Cfg<A_ROWS, STAGES, FP8>;
  constexpr int kAccBufs = FP8 ? 1 : 2;
  constexpr int kStages = STAGES;
  constexpr int kABytes = C::kABytes;
  constexpr int kStageBytes = C::kStageBytes;
  constexpr int kBarOffset = C::kBarOffset;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smem + kStages * kABytes;
  uint8_t* smSF = smem + C::kSfOffset;             // FP8: per stage, A scales then B scales
  const int kbt = a.K / (FP8 ? kKB8 : kBK);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOffset);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // fused mode: the unit queue (slot values, then the full and empty barriers)
  volatile int64_t* ring = reinterpret_cast<volatile int64_t*>(smem + (FUSED ? C::kRingOffset : 0));
  uint64_t* ufull = reinterpret_cast<uint64_t*>(smem + (FUSED ? C::kRingOffset : 0) + kRing * 8);
  uint64_t* uempty = ufull + kRing;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(drain, 1);
    if constexpr (FUSED) {
      for (int i = 0; i < kRing; ++i) {
        mbar_init(&ufull[i], 1);
        mbar_init(&uempty[i], 5);   // the MMA thread and the four epilogue warps
      }
    }
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = a.keep_weight ? policy_evict_last() : policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued[kStages] = {};
      bool ok = true;
      // Units: static round-robin (blockIdx.x, + gridDim.x, ...), or, in the
      // fused mode, tickets from a global counter: a unit is only ever taken
      // by a running CTA, so a value tile's wait for the key tiles of its M
      // tile (all with smaller tickets) never depends on a CTA that has not
      // started.  The producer hands each ticket to the MMA thread and the
      // epilogue warps through the shared-memory ring (-1: no more units).
      uint32_t rslot = 0, rphase = 0;
      auto publish = [&](int64_t v) -> bool {
        if (!mbar_wait(&uempty[rslot], rphase ^ 1u, abort_flag)) return false;
        ring[rslot] = v;
        mbar_arrive(&ufull[rslot]);
        if (++rslot == kRing) {
          rslot = 0;
          rphase ^= 1u;
        }
        return true;
      };
      int64_t u = blockIdx.x;
      if constexpr (FUSED) {
        u = atomicAdd(a.tickets, 1u);
        publish(u < a.units ? u : -1);            // a fresh ring: no wait
      }
      const int64_t first = u;
      // The weight does not depend on the kernel queued before this one (the
      // gather): the first stages of the first unit get their weight tile while
      // the gathered rows are still being written.
      int pre = 0;
      if (u < a.units) {
        int mt, nt, sp, kf, kn;
        unit_coords<FUSED>(a, u, mt, nt, sp);
        unit_kb(a, u, sp, kf, kn);
        pre = min(kStages, kn);
        for (int i = 0; i < pre; ++i) {   // fresh ring: every stage is free
          mbar_arrive_expect_tx(&full[i], kStageBytes);
          load_b<FP8>(a, tmB, smB + i * kBBytes, smSF + i * C::kSfBytes, &full[i], nt, kf + i, kbt, pol_w);
        }
      }
      grid_dependency_wait();     // the gathered rows are written by the gather kernel
      while (u < a.units && ok) {
        // the kernel queued after this one (the gate) may start arriving once
        // every CTA has begun its last unit
        if (!FUSED && u + gridDim.x >= a.units) grid_launch_dependents();
        int mt, nt, sp, kb0, kbn;
        unit_coords<FUSED>(a, u, mt, nt, sp);
        unit_kb(a, u, sp, kb0, kbn);
        for (int kb = 0; kb < kbn; ++kb) {
          uint8_t* sf = smSF + stage * C::kSfBytes;
          if (u == first && kb < pre) {
            // weight tile already in flight on this stage: add the rows
            load_a<FP8>(a, tmA, smA + stage * kABytes, sf, &full[stage], mt, kb0 + kb, kbt);
          } else {
            if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[stage], kStageBytes);
            load_a<FP8>(a, tmA, smA + stage * kABytes, sf, &full[stage], mt, kb0 + kb, kbt);
            load_b<FP8>(a, tmB, smB + stage * kBBytes, sf, &full[stage], nt, kb0 + kb, kbt, pol_w);
          }
          ++issued[stage];
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (FUSED) {
          u = atomicAdd(a.tickets, 1u);
          if (!publish(u < a.units ? u : -1)) ok = false;
        } else {
          u += gridDim.x;
        }
      }
      if (!ok) {
        raise_abort(abort_flag, a.err);
        // let every copy already issued land before the CTA can exit
        for (int s = 0; s < kStages; ++s)
          if (issued[s] > 0) mbar_wait(&full[s], (issued[s] - 1u) & 1u, nullptr, kDrainLimitNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    grid_dependency_wait();
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kBM, kBN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      uint32_t rslot = 0, rphase = 0;
      for (int64_t u = blockIdx.x;; u += gridDim.x) {
        if constexpr (FUSED) {                       // the producer's next ticket
          if (!mbar_wait(&ufull[rslot], rphase, abort_flag)) {
            ok = false;
            break;
          }
          u = ring[rslot];
          mbar_arrive(&uempty[rslot]);
          if (++rslot == kRing) {
            rslot = 0;
            rphase ^= 1u;
          }
          if (u < 0) break;
        } else {
          if (u >= a.units) break;
          if (u + gridDim.x >= a.units) grid_launch_dependents();
        }
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        int kb_first, kbn;
        unit_kb(a, u, remainder_unit(a, u) ? static_cast<int>((u - a.full_units) % a.rem_splits)
                                           : static_cast<int>(u % a.splits),
                kb_first, kbn);
        for (int kb = 0; kb < kbn; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(smA + stage * kABytes));
          const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(smB + stage * kBBytes));
          if constexpr (FP8) {
            // the stage's scales into tensor memory, then four K = 32 steps
            // (+32 bytes each) that take scale byte kk of each 32-bit column
            const uint32_t sf_col = tmem_base + kSfCol0 + static_cast<uint32_t>(stage) * kSfColsPerStage;
            const uint32_t sf_smem = smem_u32(smSF + stage * C::kSfBytes);
            tmem_cp_32x128b_warpx4(sf_col, sdesc_rows16(sf_smem));
            tmem_cp_32x128b_warpx4(sf_col + 4, sdesc_rows16(sf_smem + kSfaBytes));
            tmem_cp_32x128b_warpx4(sf_col + 8, sdesc_rows16(sf_smem + kSfaBytes + kSfbBytes / 2));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              umma_mxf8(d_tmem, adesc + 2ull * kk, bdesc + 2ull * kk, idesc_mxf8_e4m3(kBM, kBN, kk), sf_col,
                        sf_col + 4, (kb | kk) != 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              // +32 bytes per K step of 16 bf16 = +2 in the start-address field
              umma_bf16(d_tmem, adesc + 2ull * kk, bdesc + 2ull * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
            }
          }
          umma_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        if (++acc == kAccBufs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // every MMA issued by this thread completes before the tensor memory is freed
      umma_commit(drain);
      mbar_wait(drain, 0, nullptr, kDrainLimitNs);
      if (!ok) raise_abort(abort_flag, a.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    grid_dependency_wait();   // the outputs may still be read by an earlier kernel
    const int q = warp & 3;   // tensor-memory lane quarter this warp may read
    // this warp's staging tile
    uint8_t* epi = smem + C::kEpiOffset + (warp - 2) * (FUSED ? kEpiWarpBytes : kPlainWarpBytes);
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    uint32_t rslot = 0, rphase = 0;
    for (int64_t u = blockIdx.x;; u += gridDim.x) {
      if constexpr (FUSED) {                         // the producer's next ticket
        if (!mbar_wait(&ufull[rslot], rphase, abort_flag)) {
          ok = false;
          break;
        }
        u = ring[rslot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&uempty[rslot]);
        if (++rslot == kRing) {
          rslot = 0;
          rphase ^= 1u;
        }
        if (u < 0) break;
      } else {
        if (u >= a.units) break;
        if (u + gridDim.x >= a.units) grid_launch_dependents();
      }
      int mt, nt, sp;
      unit_coords<FUSED>(a, u, mt, nt, sp);
      if constexpr (FUSED) {
        // the rows of x this warp's epilogue of the unit will read, asked of
        // the L2 now, while the unit's MMAs still run
        const int64_t mr = static_cast<int64_t>(mt) * kBM + q * 32 + lane;
        if (mr < a.M) {
          if (nt < a.key_n_tiles) {
            const int s = nt * kBN / a.dim, d0 = nt * kBN - s * a.dim;
            prefetch_l2(a.x + (mr * a.hc + s) * a.dim + d0, kBN * 2);
          } else {
            const int d0 = (nt - a.key_n_tiles) * kBN;
            for (int s = 0; s < a.hc; ++s) prefetch_l2(a.x + (mr * a.hc + s) * a.dim + d0, kBN * 2);
          }
        }
      }
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int64_t m = static_cast<int64_t>(mt) * kBM + q * 32 + lane;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kBN);
      bool released = false;                         // the accumulator already handed back
      if constexpr (!FUSED) {
        if (FP8 && a.out_mode == kOutBf16 && !remainder_unit(a, u)) {
          bf16_epilogue_release_first(a, t_row, m - lane, nt, lane, smem_u32(epi), &tempty[acc]);
          released = true;
        } else if (remainder_unit(a, u)) {
          // remainder unit j (tile j / rem_splits, K range sp): its fp32 sums go to
          // the workspace; launch_reduce_remainder adds the ranges up afterwards
          const int64_t j = u - a.full_units;
          plain_epilogue<BULK>(a, t_row, m - lane, nt, sp, lane, smem_u32(epi), a.rem_ws + (j * kBM + q * 32) * kBN,
                               kBN);
        } else {
          plain_epilogue<BULK>(a, t_row, m - lane, nt, sp, lane, smem_u32(epi));
        }
      } else if (nt < a.key_n_tiles) {
        fused_key_epilogue(a, t_row, m, nt * kBN, lane, reinterpret_cast<float*>(epi));
        fused_key_publish(a, m, mt, q, lane);
      } else if (!fused_value_epilogue(a, t_row, m, mt, q, nt * kBN, lane, abort_flag, epi)) {
        ok = false;
        break;
      }
      if (!released) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
      }
      if (++acc == kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (!ok && lane == 0) raise_abort(abort_flag, a.err);
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
  if constexpr (FUSED) {
    // Every CTA has taken its last ticket (before the barrier above); the last
    // CTA to get here puts the ticket counter back to 0 for the next launch.
    // The fused kernel never triggers its dependents early (no
    // griddepcontrol.launch_dependents): the next kernel in the stream, which
    // may be the next fused projection taking tickets before its own
    // dependency wait, launches only once every CTA, and so the reset, is done.
    if (threadIdx.x == 0 && atom_acq_rel_add_u32(a.tickets + 1, 1u) == gridDim.x - 1) {
      atomicExch(a.tickets, 0u);
      atomicExch(a.tickets + 1, 0u);
    }
  }
}

// ---------------------------------------------------------------- CTA-pair projection
// The projection for bf16 kv without split-K on pairs of CTAs (clusters of
// two, neighbouring SMs) with tcgen05.mma.cta_group::2:
//  * a unit is a 256 x 256 output tile -- two M tiles by one N tile -- over
//    the whole K;
//  * CTA r of the pair loads rows r*128 .. r*128+127 of the unit's A rows and
//    rows r*128 .. of its weight tile (the first or the second 16 KB of the
//    packed 32 KB tile) into its own shared memory, so each SM keeps and
//    reads half the weight bytes per FLOP of the one-CTA kernel (the MMA
//    takes the other half from the peer);
//  * both CTAs' tensor copies count their bytes on the even CTA's stage
//    barrier (the cta_group::2 form of the copy), so the even CTA's MMA thread
//    issues the pair's MMAs as soon as a stage has landed in both, and each of
//    its commits arrives on the barriers of both CTAs at once;
//  * each CTA's epilogue drains its own tensor memory (its 128 rows) like the
//    one-CTA kernel and reports the accumulator free to the even CTA.
// Every wait is bounded, as in wkv_gemm_kernel.
// Shared memory of the pair kernel.  The fused mode keeps five operand stages
// (six otherwise) to make room for each epilogue warp's x staging buffers.
constexpr int kXBufs = 3;                       // x staging buffers per epilogue warp (fused)
constexpr int kXBufBytes = 4096;                // one x chunk: 32 tokens x 64 channels of one stream
template <bool FUSED>
struct PairCfgT {
  static constexpr int kStages = FUSED ? 5 : 6;
  static constexpr int kABytes = kBM * kBK * 2;                  // 16 KB: 128 rows of A
  static constexpr int kBHalf = kBBytes / 2;                     // 16 KB: 128 rows of the weight tile
  static constexpr int kStageBytes = kABytes + kBHalf;
  static constexpr int kXOffset = kStages * kStageBytes;         // 1024-byte aligned
  static constexpr int kBarOffset = kXOffset + (FUSED ? 4 * kXBufs * kXBufBytes : 0);
  // full, empty, tfull, tempty, drain; fused: each epilogue warp's x buffers
  static constexpr int kNumBars = 2 * kStages + 2 + 2 + 1 + (FUSED ? 4 * kXBufs : 0);
  static constexpr int kEpiOffset = kBarOffset + 256;
  // plain: the epilogue's staging tile; fused: a key tile's 256 weight products
  static constexpr int kEpiWarp = FUSED ? 1024 : kPlainWarpBytes;
  static constexpr size_t kRingOffset = kEpiOffset + 4 * kEpiWarp;   // fused: the CTA's unit queue
  static constexpr size_t kSmemBytes = 1024 + kRingOffset + (FUSED ? kRingBytes : 0);
  static_assert(kNumBars * 8 + 8 <= 256, "barrier area");
  static_assert(kXOffset % 1024 == 0 && kXBufBytes % 1024 == 0, "x buffers take the 128-byte swizzle");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};
using PairCfg = PairCfgT<false>;
using PairFusedCfg = PairCfgT<true>;

// The tensor maps of the fused pair epilogue, over x and out viewed as
// [M][hc][dim] bf16: boxes of 32 tokens x 1 stream x 64 channels (4 KB, one
// 128-byte row per token) with the 128-byte swizzle.
struct PairXMaps {
  CUtensorMap x, out;
};

// Pair unit u -> (M pair p: M tiles 2p, 2p+1; N tile nt), rasterised in
// groups of group_m M pairs, M fastest inside a group.
__device__ __forceinline__ void pair_coords(const GemmArgs& a, int64_t u, int& mp, int& nt) {
  const int m_pairs = (a.m_tiles + 1) >> 1;
  const int64_t group_units = static_cast<int64_t>(a.group_m) * a.n_tiles;
  const int64_t g = u / group_units;
  const int64_t r = u - g * group_units;
  const int gm0 = static_cast<int>(g) * a.group_m;
  const int gm = min(a.group_m, m_pairs - gm0);
  nt = static_cast<int>(r / gm);
  mp = gm0 + static_cast<int>(r % gm);
}

// Pair unit u: its tile (mp, nt) and K blocks [kb0, kb0 + kbn).  Units past
// full_units are the remainder: the last rem_tiles pair tiles of the raster
// order, each cut into rem_splits K ranges of rem_kb blocks (range j % rem_splits
// of tile j / rem_splits); returns that j, or -1 for a whole tile.
__device__ __forceinline__ int64_t pair_unit(const GemmArgs& a, int64_t u, int kbt, int& mp, int& nt, int& kb0,
                                             int& kbn) {
  if (a.rem_splits > 0 && u >= a.full_units) {
    const int64_t j = u - a.full_units;
    pair_coords(a, a.full_units + j / a.rem_splits, mp, nt);
    kb0 = static_cast<int>(j % a.rem_splits) * a.rem_kb;
    kbn = a.rem_kb;
    return j;
  }
  pair_coords(a, u, mp, nt);
  kb0 = 0;
  kbn = kbt;
  return -1;
}

// Pair unit u of the fused mode: the fused order of fused_coords over M pairs,
// whole K.
template <bool FUSED>
__device__ __forceinline__ int64_t pair_unit_of(const GemmArgs& a, int64_t u, int kbt, int& mp, int& nt, int& kb0,
                                                int& kbn) {
  if constexpr (FUSED) {
    fused_coords(a, u, (a.m_tiles + 1) >> 1, mp, nt);
    kb0 = 0;
    kbn = kbt;
    return -1;
  }
  return pair_unit(a, u, kbt, mp, nt, kb0, kbn);
}

// A fused-pair epilogue warp's x staging: kXBufs buffers filled in turn by
// tensor copies that lane 0 issues; every lane waits for a chunk in the order
// issued.  `issued` is lane 0's count, `used` every lane's.  The copies are
// L2 evict-first: the key tiles read each element of x once, and by the time
// the value tiles read it again (a group of key tiles later) it is gone from
// the L2 either way, so x should not push the weight and the gathered rows,
// which are read over and over, out of it (full_2x8192: DRAM reads of the
// kernel 5.40 -> 4.77 GB, the time the same).
struct XStage {
  uint8_t* base;
  uint64_t* bars;
  uint32_t issued;
  uint32_t used;
  __device__ __forceinline__ void issue(const CUtensorMap* map, uint32_t bytes, int32_t x, int32_t y, int32_t z) {
    const uint32_t b = issued % kXBufs;
    mbar_arrive_expect_tx(&bars[b], bytes);
    tma_load_3d_hint(base + b * kXBufBytes, map, &bars[b], x, y, z, policy_evict_first());
    ++issued;
  }
  // the next chunk's shared address, once it has landed; false if the wait ran out
  __device__ __forceinline__ bool wait(volatile int* abort_flag, uint32_t& addr) {
    const uint32_t b = used % kXBufs;
    const bool ok = mbar_wait(&bars[b], (used / kXBufs) & 1u, abort_flag);
    addr = smem_u32(base + b * kXBufBytes);
    ++used;
    return __all_sync(0xFFFFFFFFu, ok);
  }
  // lane 0: let every copy still in flight land (leaving early)
  __device__ __forceinline__ void drain() {
    for (uint32_t k = used; k < issued; ++k)
      mbar_wait(&bars[k % kXBufs], (k / kXBufs) & 1u, nullptr, kDrainLimitNs);
    used = issued;
  }
};

// Byte b of a staged box image sits at b with its 16-byte chunk index
// (bits 4-6) xor-ed with bits 7-9: the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz128(uint32_t b) { return b ^ (((b >> 7) & 7u) << 4); }

constexpr int kChunkCols = 64;                  // channels of one staged x chunk

// Key tile of the fused pair epilogue: fused_key_epilogue's sums, in its order,
// with row m's hidden state read from the staged chunks (the block's 4 chunks
// of 64 channels; chunks 0 and 1 issued at the unit's start, chunk c + 2 once
// chunk c is read).  Lane = row.
__device__ __forceinline__ bool pair_key_epilogue(const GemmArgs& a, const CUtensorMap* tmx, uint32_t t_row,
                                                  int64_t m0, int n0, int lane, float* wsm, XStage& xs,
                                                  volatile int* abort_flag) {
  const int s = n0 / a.dim;
  const int d0 = n0 - s * a.dim;
  const int64_t m = m0 + lane;
  const bool active = m < a.M && (a.mask == nullptr || a.mask[m] != 0);
  {
    const float4* wg = reinterpret_cast<const float4*>(a.wprod + static_cast<int64_t>(s) * a.dim + d0) + 2 * lane;
    reinterpret_cast<float4*>(wsm)[2 * lane] = __ldg(wg);
    reinterpret_cast<float4*>(wsm)[2 * lane + 1] = __ldg(wg + 1);
    __syncwarp();
  }
  float th[16], tk[16], td[16];   // the butterfly after its first step (registers: the loop is unrolled)
#pragma unroll
  for (int c = 0; c < kBN / kChunkCols; ++c) {
    uint32_t xb;
    if (!xs.wait(abort_flag, xb)) return false;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * kChunkCols + half * 32), r);
      tmem_ld_wait();
      if (active) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int j = 4 * half + g;                  // 16-byte chunk of the row's 128 bytes
          const int l = 8 * c + j;                     // group index in the block
          float h[8];
          unpack8_bf16(ld_shared_v4(xb + swz128(static_cast<uint32_t>(lane * 128 + j * 16))), h);
          const float4 w0 = reinterpret_cast<const float4*>(wsm)[2 * l];
          const float4 w1 = reinterpret_cast<const float4*>(wsm)[2 * l + 1];
          const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
          float sh = 0.0f, sk = 0.0f, sd = 0.0f;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float k = round_bf16(__uint_as_float(r[8 * g + e]));
            sh = fmaf(h[e], h[e], sh);
            sk = fmaf(k, k, sk);
            sd = fmaf(__fmul_rn(h[e], w[e]), k, sd);
          }
          if (l < 16) {
            th[l] = sh; tk[l] = sk; td[l] = sd;
          } else {                                     // butterfly step 16
            th[l - 16] = th[l - 16] + sh; tk[l - 16] = tk[l - 16] + sk; td[l - 16] = td[l - 16] + sd;
          }
        }
      }
    }
    __syncwarp();                                      // every lane has read the chunk
    if (lane == 0 && c + 2 < kBN / kChunkCols)
      xs.issue(tmx, kXBufBytes, d0 + (c + 2) * kChunkCols, s, static_cast<int32_t>(m0));
  }
  if (active) {
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) {
#pragma unroll
      for (int l = 0; l < off; ++l) {
        th[l] = th[l] + th[l + off]; tk[l] = tk[l] + tk[l + off]; td[l] = td[l] + td[l + off];
      }
    }
    const int nblk = a.dim / kBN;
    reinterpret_cast<float4*>(a.gsum)[(m * a.hc + s) * nblk + d0 / kBN] = make_float4(th[0], tk[0], td[0], 0.0f);
  }
  return true;
}

// Value tile of the fused pair epilogue: once the gates of the warp's 32 rows
// are ready, out = h + gate * value, 64 channels of one stream per staged
// chunk (chunk n: channels 64 (n / hc) .., stream n % hc), computed in place in
// the chunk and written back by a tensor store (tokens past M are not
// written; a masked token's row goes back as it came, x itself).  Lane = row.
// Returns false if a wait ran out.
__device__ __forceinline__ bool pair_value_epilogue(const GemmArgs& a, const CUtensorMap* tmx, const CUtensorMap* tmo,
                                                    uint32_t t_row, int64_t m0, int mt, int q, int n0, int lane,
                                                    XStage& xs, volatile int* abort_flag) {
  const int d0 = n0 - a.hc * a.dim;
  bool ok = true;
  if (lane == 0) {
    const unsigned long long t0 = globaltimer_ns();
    while (ld_acquire_u32(a.counters + mt * 8 + 4 + q) == 0u) {
      if (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) {
        ok = false;
        break;
      }
      __nanosleep(64);
    }
  }
  ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
  if (!ok) return false;
  __threadfence();
  const int64_t m = m0 + lane;
  const bool mix = m < a.M && (a.mask == nullptr || a.mask[m] != 0);
  float4 gv = make_float4(0.f, 0.f, 0.f, 0.f);
  if (mix) gv = __ldcg(reinterpret_cast<const float4*>(a.gates) + m);
  const float gs[kMaxStreams] = {gv.x, gv.y, gv.z, gv.w};
  const int nch = (kBN / kChunkCols) * a.hc;
#pragma unroll 1
  for (int c = 0; c < kBN / kChunkCols; ++c) {
    float v[kChunkCols];                               // kv as the projection rounds it
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * kChunkCols + half * 32), r);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) v[32 * half + e] = round_bf16(__uint_as_float(r[e]));
    }
#pragma unroll
    for (int s = 0; s < kMaxStreams; ++s) {
      if (s >= a.hc) break;
      const int n = c * a.hc + s;
      uint32_t xb;
      if (!xs.wait(abort_flag, xb)) return false;
      if (mix) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t addr = xb + swz128(static_cast<uint32_t>(lane * 128 + j * 16));
          float h[8];
          unpack8_bf16(ld_shared_v4(addr), h);
          const float* vv = v + 8 * j;
          uint4 o;
          o.x = pack_bf16x2(fmaf(gs[s], vv[0], h[0]), fmaf(gs[s], vv[1], h[1]));
          o.y = pack_bf16x2(fmaf(gs[s], vv[2], h[2]), fmaf(gs[s], vv[3], h[3]));
          o.z = pack_bf16x2(fmaf(gs[s], vv[4], h[4]), fmaf(gs[s], vv[5], h[5]));
          o.w = pack_bf16x2(fmaf(gs[s], vv[6], h[6]), fmaf(gs[s], vv[7], h[7]));
          st_shared_v4(addr, o);
        }
      }
      fence_proxy_async_shared();                      // the chunk's new bytes, for the tensor store
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(tmo, xb, d0 + c * kChunkCols, s, static_cast<int32_t>(m0));
        bulk_commit();
        if (n + 2 < nch) {
          const int n2 = n + 2;
          bulk_wait_read_but_one();                    // chunk n - 1's store has read the buffer chunk n + 2 takes
          xs.issue(tmx, kXBufBytes, d0 + (n2 / a.hc) * kChunkCols, n2 % a.hc, static_cast<int32_t>(m0));
        }
      }
    }
  }
  return true;
}

// FUSED: the gate epilogue of wkv_gemm_kernel, on the pair's tiles.  Units
// then come from the work-ticket counter: the even CTA's producer takes a
// ticket and writes it into the unit queue of both CTAs (its own and, through
// the cluster window, the odd CTA's); the even CTA's queue slot is free once
// its MMA thread and epilogue warps and the odd CTA's producer and epilogue
// warps have read it (10 arrivals on the even CTA's barrier).  Each CTA's
// epilogue treats its 128 rows -- M tile 2p + rank -- as one M tile of the
// one-CTA fused kernel, with x staged in shared memory by tensor copies (xm)
// and the output written by tensor stores.
template <bool BULK, bool FUSED>
__global__ void __launch_bounds__(kGemmThreads, 1)
    wkv_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                         const __grid_constant__ PairXMaps xm, const GemmArgs a) {
  using C = PairCfgT<FUSED>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smA = smem;                             // stage s at s * kABytes
  uint8_t* smB = smem + S * C::kABytes;            // stage s at s * kBHalf
  const int kbt = a.K / kBK;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  uint64_t* full = bars;                           // even CTA: the stage landed in both CTAs
  uint64_t* empty = bars + S;                      // the pair's MMAs are done with the stage
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = tfull + 2;                    // even CTA: 8 epilogue warps of the pair
  uint64_t* drain = tempty + 2;
  uint64_t* xbars = drain + 1;                     // fused: kXBufs per epilogue warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xbars + (FUSED ? 4 * kXBufs : 0));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // fused mode: the unit queue (slot values, then the full and empty barriers)
  volatile int64_t* ring = reinterpret_cast<volatile int64_t*>(smem + (FUSED ? C::kRingOffset : 0));
  uint64_t* ufull = reinterpret_cast<uint64_t*>(smem + (FUSED ? C::kRingOffset : 0) + kRing * 8);
  uint64_t* uempty = ufull + kRing;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int64_t pair = blockIdx.x >> 1;
  const int64_t npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 8);
    }
    mbar_init(drain, 1);
    if constexpr (FUSED) {
      for (int i = 0; i < kRing; ++i) {
        mbar_init(&ufull[i], 1);
        mbar_init(&uempty[i], 10);
      }
      for (int i = 0; i < 4 * kXBufs; ++i) mbar_init(&xbars[i], 1);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmW);
    if constexpr (FUSED) {
      tma_prefetch_desc(&xm.x);
      tma_prefetch_desc(&xm.out);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_arrive();                                // both CTAs' barriers exist before any copy counts on them
  cluster_wait();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // fused mode: read the next unit from this CTA's queue and free the slot
  // (on the even CTA's barrier); -2 if the wait ran out
  uint32_t rslot = 0, rphase = 0;
  auto next_queued = [&](bool one_lane) -> int64_t {
    const bool got = rank == 0 ? mbar_wait(&ufull[rslot], rphase, abort_flag)
                               : mbar_wait_cluster(&ufull[rslot], rphase, abort_flag);
    const int64_t v = got ? ring[rslot] : -2;
    if (one_lane) __syncwarp();
    if (got && (!one_lane || lane == 0)) {
      if (rank == 0) mbar_arrive(&uempty[rslot]);
      else mbar_arrive_remote(mapa_shared(&uempty[rslot], 0));
    }
    if (++rslot == kRing) {
      rslot = 0;
      rphase ^= 1u;
    }
    return v;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      const uint64_t pol_w = a.keep_weight ? policy_evict_last() : policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      uint32_t full_even[S];                       // the even CTA's stage barriers
      for (int i = 0; i < S; ++i) full_even[i] = mapa_shared(&full[i], 0);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued[S] = {};
      bool ok = true;
      // fused mode: the even CTA takes the pair's tickets and queues them in
      // both CTAs (-1: no more units); the odd CTA reads its queue
      auto take = [&]() -> int64_t {
        if (rank != 0) return next_queued(false);
        if (!mbar_wait_cluster(&uempty[rslot], rphase ^ 1u, abort_flag)) return -2;
        const uint32_t t = atomicAdd(a.tickets, 1u);
        const int64_t v = t < a.units ? static_cast<int64_t>(t) : -1;
        ring[rslot] = v;
        st_cluster_s64(mapa_shared(const_cast<int64_t*>(&ring[rslot]), 1), v);
        mbar_arrive(&ufull[rslot]);
        mbar_arrive_remote(mapa_shared(&ufull[rslot], 1));
        if (++rslot == kRing) {
          rslot = 0;
          rphase ^= 1u;
        }
        return v;
      };
      int64_t u = pair;
      if constexpr (FUSED) {
        u = take();
        if (u == -2) ok = false;
      }
      const int64_t first = u;
      int pre = 0;
      if (ok && u >= 0 && u < a.units) {           // the weight halves of the first stages, before the wait
        int mp, nt, kb0, kbn;
        pair_unit_of<FUSED>(a, u, kbt, mp, nt, kb0, kbn);
        pre = min(S, kbn);
        for (int i = 0; i < pre; ++i) {
          if (rank == 0) mbar_arrive_expect_tx(&full[i], 2 * C::kStageBytes);
          tma_load_2d_pair(smB + i * C::kBHalf, &tmW, full_even[i], 0,
                           (nt * kbt + kb0 + i) * kBN + static_cast<int32_t>(rank) * kBM, pol_w);
        }
      }
      grid_dependency_wait();                      // the gathered rows are written by the gather kernel
      while (ok && u >= 0 && u < a.units) {
        if (!FUSED && u + npairs >= a.units) grid_launch_dependents();
        int mp, nt, kb0, kbn;
        pair_unit_of<FUSED>(a, u, kbt, mp, nt, kb0, kbn);
        const int32_t row0 = mp * (2 * kBM) + static_cast<int32_t>(rank) * kBM;
        for (int kb = 0; kb < kbn; ++kb) {
          if (!(u == first && kb < pre)) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * C::kStageBytes);
            tma_load_2d_pair(smB + stage * C::kBHalf, &tmW, full_even[stage], 0,
                             (nt * kbt + kb0 + kb) * kBN + static_cast<int32_t>(rank) * kBM, pol_w);
          }
          tma_load_2d_pair(smA + stage * C::kABytes, &tmA, full_even[stage], (kb0 + kb) * kBK, row0, pol_a);
          ++issued[stage];
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (FUSED) {
          u = take();
          if (u == -2) ok = false;
        } else {
          u += npairs;
        }
      }
      if (!ok) {
        raise_abort(abort_flag, a.err);
        // the even CTA waits for the copies in flight (they count on its
        // barriers).  The odd CTA's are among them: both producers refill a
        // stage only once its free barrier completes, and one multicast commit
        // completes it in both CTAs at once; a wait runs out only after the
        // MMA thread has stopped committing, so both have refilled the same
        // stages.
        if (rank == 0)
          for (int i = 0; i < S; ++i)
            if (issued[i] > 0) mbar_wait(&full[i], (issued[i] - 1u) & 1u, nullptr, kDrainLimitNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    grid_dependency_wait();
    if (rank == 0 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer (even CTA)
      const uint32_t idesc = idesc_bf16_f32(2 * kBM, kBN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int64_t u = pair;; u += npairs) {
        if constexpr (FUSED) {
          u = next_queued(false);
          if (u == -2) ok = false;
          if (u < 0) break;
        } else {
          if (u >= a.units) break;
          if (u + npairs >= a.units) grid_launch_dependents();
        }
        if (!mbar_wait_cluster(&tempty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        int mp, nt, kb0, kbn;
        pair_unit_of<FUSED>(a, u, kbt, mp, nt, kb0, kbn);
        for (int kb = 0; kb < kbn; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(smA + stage * C::kABytes));
          const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(smB + stage * C::kBHalf));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16_pair(d_tmem, adesc + 2ull * kk, bdesc + 2ull * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
          umma_commit_pair(&empty[stage], 3);      // the stage is free in both CTAs
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(&tfull[acc], 3);          // the accumulator is ready in both CTAs
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // every MMA issued completes before either CTA frees its tensor memory
      umma_commit_pair(drain, 1);
      mbar_wait(drain, 0, nullptr, kDrainLimitNs);
      if (!ok) raise_abort(abort_flag, a.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    grid_dependency_wait();
    const int q = warp & 3;
    uint8_t* epi = smem + C::kEpiOffset + (warp - 2) * C::kEpiWarp;
    const uint32_t tempty_even[2] = {mapa_shared(&tempty[0], 0), mapa_shared(&tempty[1], 0)};
    XStage xs{smem + C::kXOffset + (warp - 2) * kXBufs * kXBufBytes, xbars + (warp - 2) * kXBufs, 0u, 0u};
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int64_t u = pair;; u += npairs) {
      if constexpr (FUSED) {
        u = next_queued(true);
        if (u == -2) ok = false;
        if (u < 0) break;
      } else {
        if (u >= a.units) break;
        if (u + npairs >= a.units) grid_launch_dependents();
      }
      int mp, nt, kb0, kbn;
      const int64_t j = pair_unit_of<FUSED>(a, u, kbt, mp, nt, kb0, kbn);
      const int mt = 2 * mp + static_cast<int>(rank);
      const int64_t m0 = static_cast<int64_t>(mt) * kBM + q * 32;
      // fused: whether this warp holds rows (the odd CTA of a last pair over an
      // odd number of M tiles holds none, and the last M tile may end early)
      const bool rows = mt < a.m_tiles && m0 < a.M;
      if constexpr (FUSED) {
        if (rows) {
          // the unit's first two chunks of x into the staging buffers, while
          // the unit's MMAs run
          const bool key = nt < a.key_n_tiles;
          const int s = key ? nt * kBN / a.dim : 0;
          const int d0 = key ? nt * kBN - s * a.dim : (nt - a.key_n_tiles) * kBN;
          if (lane == 0) {
            bulk_wait_read_all();                  // the last unit's stores have read their buffers
            for (int n = 0; n < 2; ++n) {          // key: chunk n of stream s; value: chunk n of the streams
              if (key) xs.issue(&xm.x, kXBufBytes, d0 + n * kChunkCols, s, static_cast<int32_t>(m0));
              else xs.issue(&xm.x, kXBufBytes, d0 + (n / a.hc) * kChunkCols, n % a.hc, static_cast<int32_t>(m0));
            }
          }
        }
      }
      if (!mbar_wait_cluster(&tfull[acc], acc_phase, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kBN);
      if constexpr (FUSED) {
        if (rows) {
          if (nt < a.key_n_tiles) {
            if (!pair_key_epilogue(a, &xm.x, t_row, m0, nt * kBN, lane, reinterpret_cast<float*>(epi), xs,
                                   abort_flag)) {
              ok = false;
              break;
            }
            fused_key_publish(a, m0 + lane, mt, q, lane);
          } else if (!pair_value_epilogue(a, &xm.x, &xm.out, t_row, m0, mt, q, nt * kBN, lane, xs, abort_flag)) {
            ok = false;
            break;
          }
        }
      } else if (j >= 0) {
        // remainder range j % rem_splits of tile j / rem_splits: this CTA's
        // 128 rows of fp32 sums to the workspace, [tile][range][CTA][128][256]
        float* ws = a.rem_ws + ((j * 2 + rank) * kBM + q * 32) * kBN;
        plain_epilogue<false>(a, t_row, m0, nt, 0, lane, smem_u32(epi), ws, kBN);
      } else {
        plain_epilogue<BULK>(a, t_row, m0, nt, 0, lane, smem_u32(epi));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(&tempty[acc]);
        else mbar_arrive_remote(tempty_even[acc]);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (!ok && lane == 0) raise_abort(abort_flag, a.err);
    if constexpr (FUSED) {
      if (lane == 0) {
        xs.drain();                                // copies still in flight (leaving early)
        bulk_wait_all();                           // the tensor stores are done
      }
    }
    __syncwarp();
  }

  // neither CTA frees its tensor memory before the pair's MMAs and both
  // epilogues are done
  tc_fence_before();
  __syncthreads();
  cluster_arrive();
  cluster_wait();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
  if constexpr (FUSED) {
    // every even CTA has taken its last ticket; the last CTA here resets the
    // counter for the next launch (no early launch of dependents, as in
    // wkv_gemm_kernel's fused mode)
    if (threadIdx.x == 0 && atom_acq_rel_add_u32(a.tickets + 1, 1u) == gridDim.x - 1) {
      atomicExch(a.tickets, 0u);
      atomicExch(a.tickets + 1, 0u);
    }
  }
}

template <int A_ROWS, int STAGES>
cudaError_t set_smem_attr() {
  using C = Cfg<A_ROWS, STAGES>;
  using C8 = Cfg<A_ROWS, STAGES, true>;
  cudaError_t e = cudaFuncSetAttribute(wkv_gemm_kernel<A_ROWS, STAGES, false, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmemBytes));
  if (e == cudaSuccess && C::kCanFuse)
    e = cudaFuncSetAttribute(wkv_gemm_kernel<A_ROWS, STAGES, true, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmemFused));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(wkv_gemm_kernel<A_ROWS, STAGES, false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C8::kSmemBytes));
  if constexpr (A_ROWS == kBM) {
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(wkv_gemm_kernel<A_ROWS, STAGES, false, false, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmemBytes));
  }
  return e;
}

template <int A_ROWS, int STAGES>
cudaError_t launch_variant(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a, int ctas,
                           cudaStream_t stream) {
  using C = Cfg<A_ROWS, STAGES>;
  const bool fused = a.out_mode == kOutFused;
  if (a.fp8) {
    if (fused || a.wpack == nullptr || a.sfa == nullptr || a.sfb == nullptr) return cudaErrorInvalidConfiguration;
    return launch_pdl(wkv_gemm_kernel<A_ROWS, STAGES, false, true>, dim3(static_cast<unsigned>(ctas)),
                      dim3(kGemmThreads), Cfg<A_ROWS, STAGES, true>::kSmemBytes, stream, 1, tmA, tmB, a);
  }
  if constexpr (A_ROWS == kBM) {                    // bulk-copy epilogue: large bf16 batches only
    if (!fused && a.bulk_epilogue)
      return launch_pdl(wkv_gemm_kernel<A_ROWS, STAGES, false, false, true>, dim3(static_cast<unsigned>(ctas)),
                        dim3(kGemmThreads), C::kSmemBytes, stream, 1, tmA, tmB, a);
  }
  if (!fused)
    return launch_pdl(wkv_gemm_kernel<A_ROWS, STAGES, false, false>, dim3(static_cast<unsigned>(ctas)),
                      dim3(kGemmThreads), C::kSmemBytes, stream, 1, tmA, tmB, a);
  if (!C::kCanFuse) return cudaErrorInvalidConfiguration;
  return launch_pdl(wkv_gemm_kernel<A_ROWS, STAGES, true, false>, dim3(static_cast<unsigned>(ctas)),
                    dim3(kGemmThreads), C::kSmemFused, stream, 1, tmA, tmB, a);
}

// One thread per 16-byte chunk of the packed weight: chunk p of row r of a tile
// holds the row's logical chunk p ^ (r % 8), the 128-byte swizzle.
__global__ void __launch_bounds__(256) pack_wkv_kernel(const uint16_t* __restrict__ w, int64_t K, int64_t chunks,
                                                       uint4* __restrict__ out) {
  const int64_t kb_total = K / kBK;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < chunks;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tile = i >> 11;                     // 2048 chunks of 16 bytes per 32 KB tile
    const int r = static_cast<int>((i >> 3) & 255);
    const int c = static_cast<int>(i & 7) ^ (r & 7);
    const int64_t nt = tile / kb_total;
    const int64_t kb = tile - nt * kb_total;
    const int64_t n = nt * kBN + r;
    out[i] = __ldg(reinterpret_cast<const uint4*>(w + n * K + kb * kBK + c * 8));
  }
}

// One thread per byte of the packed FP8 weight scales: tile (n_tile, k_block)
// holds 1 KB, two 512-byte blocks (rows 0-127, 128-255 of the tile); in a
// block, byte 16*l + 4*q + j is the scale of K-block j of row l + 32*q.
__global__ void __launch_bounds__(256) pack_sfb_kernel(const uint8_t* __restrict__ sc, int64_t kb_total,
                                                       int64_t bytes, uint8_t* __restrict__ out) {
  const int64_t per_row = kb_total * 4;               // scales per weight row (K / 32)
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < bytes;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tile = i >> 10;
    const int b = static_cast<int>(i & 1023);
    const int half = b >> 9;
    const int l = (b >> 4) & 31;
    const int q = (b >> 2) & 3;
    const int j = b & 3;
    const int64_t nt = tile / kb_total;
    const int64_t kb = tile - nt * kb_total;
    const int64_t n = nt * kBN + half * 128 + q * 32 + l;
    out[i] = sc[n * per_row + kb * 4 + j];
  }
}

// kv of the remainder tiles: thread (tile, row, lane) adds the tile row's 8
// columns 8*lane .. over the K ranges in range order and rounds to bf16.
__global__ void __launch_bounds__(256) reduce_remainder_kernel(const GemmArgs a) {
  grid_dependency_wait();        // the projection wrote the ranges' sums
  grid_launch_dependents();
  // one-CTA tiles: workspace [tile][range][128][256]; CTA pairs: 256-row
  // tiles, [tile][range][CTA][128][256] (range r of a tile is 2 * 128 rows on)
  const int tile_rows = a.pair ? 2 * kBM : kBM;
  const int64_t total = static_cast<int64_t>(a.rem_tiles) * tile_rows * 32;
  const int64_t range_stride = static_cast<int64_t>(tile_rows) * kBN;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int lane = static_cast<int>(i & 31);
    const int row = static_cast<int>((i >> 5) % tile_rows);
    const int64_t tr = (i >> 5) / tile_rows;
    int mt, nt;
    int64_t m;
    if (a.pair) {
      pair_coords(a, a.full_units + tr, mt, nt);
      m = static_cast<int64_t>(mt) * (2 * kBM) + row;
    } else {
      raster(a, static_cast<int64_t>(a.m_tiles) * a.n_tiles - a.rem_tiles + tr, a.n_tiles, mt, nt);
      m = static_cast<int64_t>(mt) * kBM + row;
    }
    if (m >= a.M) continue;
    const float* p = a.rem_ws + (tr * a.rem_splits * tile_rows + row) * kBN + lane * 8;
    float4 lo = __ldcg(reinterpret_cast<const float4*>(p)), hi = __ldcg(reinterpret_cast<const float4*>(p) + 1);
    for (int s = 1; s < a.rem_splits; ++s) {
      const float4* ps = reinterpret_cast<const float4*>(p + s * range_stride);
      const float4 c = __ldcg(ps), d = __ldcg(ps + 1);
      lo.x += c.x; lo.y += c.y; lo.z += c.z; lo.w += c.w;
      hi.x += d.x; hi.y += d.y; hi.z += d.z; hi.w += d.w;
    }
    *reinterpret_cast<uint4*>(a.kv + m * a.N + nt * kBN + lane * 8) =
        make_uint4(pack_bf16x2(lo.x, lo.y), pack_bf16x2(lo.z, lo.w), pack_bf16x2(hi.x, hi.y), pack_bf16x2(hi.z, hi.w));
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

int gemm_a_rows(int64_t M) { return M <= 32 ? 32 : (M <= 64 ? 64 : kBM); }

bool gemm_can_fuse(int64_t M) {
  const int ar = gemm_a_rows(M);
  return ar == 32 ? Cfg<32, 5>::kCanFuse : (ar == 64 ? Cfg<64, 5>::kCanFuse : Cfg<128, 4>::kCanFuse);
}

bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_u8(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kKB8), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t gemm_prepare() {
  cudaError_t e = set_smem_attr<128, 4>();
  if (e == cudaSuccess) e = set_smem_attr<64, 5>();
  if (e == cudaSuccess) e = set_smem_attr<32, 5>();
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(wkv_gemm_pair_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(PairCfg::kSmemBytes));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(wkv_gemm_pair_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(PairCfg::kSmemBytes));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(wkv_gemm_pair_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(PairFusedCfg::kSmemBytes));
  return e;
}

int gemm_pair_slots(int num_sms) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms & ~1));
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = PairCfg::kSmemBytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, wkv_gemm_pair_kernel<false, false>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return clusters < num_sms / 2 ? clusters : num_sms / 2;
}

cudaError_t launch_pack_wkv(const uint16_t* wkv, int64_t N, int64_t K, uint8_t* packed, cudaStream_t stream) {
  if (N % kBN != 0 || K % kBK != 0) return cudaErrorInvalidValue;
  const int64_t chunks = N * K / 8;
  if (chunks == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((chunks + 255) / 256, 65536);
  pack_wkv_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(wkv, K, chunks, reinterpret_cast<uint4*>(packed));
  return cudaGetLastError();
}

cudaError_t launch_reduce_remainder(const GemmArgs& a, int num_sms, cudaStream_t stream) {
  if (a.rem_splits == 0 || a.rem_tiles == 0) return cudaSuccess;
  const int64_t total = static_cast<int64_t>(a.rem_tiles) * (a.pair ? 2 * kBM : kBM) * 32;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, static_cast<int64_t>(num_sms) * 8);
  return launch_pdl(reduce_remainder_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, 1, a);
}

cudaError_t launch_pack_sfb(const uint8_t* wkv_scale, int64_t N, int64_t K, uint8_t* packed, cudaStream_t stream) {
  if (N % kBN != 0 || K % kKB8 != 0) return cudaErrorInvalidValue;
  const int64_t bytes = N * K / 32;
  if (bytes == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((bytes + 255) / 256, 65536);
  pack_sfb_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(wkv_scale, K / kKB8, bytes, packed);
  return cudaGetLastError();
}

cudaError_t launch_gemm(const void* rows, const CUtensorMap& tmB, const GemmArgs& a, int ctas,
                        cudaStream_t stream) {
  if (a.units == 0) return cudaSuccess;
  if (a.pair) {                                     // CTA pairs: 128-row A boxes, grid of whole clusters
    // the packed weight as 128-byte rows (each 32 KB tile is 256 of them, already
    // in the swizzled order): a box of 128 rows is one CTA's half of a tile
    CUtensorMap tmA, tmW;
    auto enc = encode_fn();
    const uint64_t w_rows = static_cast<uint64_t>(a.N) * static_cast<uint64_t>(a.K / kBK);
    const cuuint64_t wdims[2] = {static_cast<cuuint64_t>(kBK), w_rows};
    const cuuint64_t wstrides[1] = {static_cast<cuuint64_t>(kBK * 2)};
    const cuuint32_t wbox[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(kBM)};
    const cuuint32_t estr[2] = {1, 1};
    const bool fused = a.out_mode == kOutFused;
    if (a.fp8 || (a.out_mode != kOutBf16 && !fused) || a.wpack == nullptr || (ctas & 1) != 0 || enc == nullptr ||
        (fused && a.rem_splits != 0) ||
        !make_tmap_bf16(&tmA, rows, static_cast<uint64_t>(a.M), static_cast<uint64_t>(a.K), kBM) ||
        enc(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint8_t*>(a.wpack), wdims, wstrides, wbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(ctas));
    PairXMaps xm;
    std::memset(&xm, 0, sizeof(xm));
    if (fused) {
      // x and out as [M][hc][dim] bf16, boxes of 64 channels x 1 stream x 32
      // tokens: 128 bytes per token, the 128-byte swizzle's row (the box's
      // inner extent is exactly the swizzle span)
      const cuuint64_t xdims[3] = {static_cast<cuuint64_t>(a.dim), static_cast<cuuint64_t>(a.hc),
                                   static_cast<cuuint64_t>(a.M)};
      const cuuint64_t xstrides[2] = {static_cast<cuuint64_t>(a.dim) * 2, static_cast<cuuint64_t>(a.hc) * a.dim * 2};
      const cuuint32_t box[3] = {static_cast<cuuint32_t>(kChunkCols), 1, 32};
      const cuuint32_t estr3[3] = {1, 1, 1};
      auto enc3 = [&](CUtensorMap* m, const void* base) {
        return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), xdims, xstrides, box, estr3,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
      };
      if (a.hc < 1 || a.hc > kMaxStreams || a.dim % kBN != 0 || !enc3(&xm.x, a.x) || !enc3(&xm.out, a.out))
        return cudaErrorInvalidValue;
      return launch_pdl(wkv_gemm_pair_kernel<false, true>, grid, dim3(kGemmThreads), PairFusedCfg::kSmemBytes, stream,
                        2, tmA, tmW, xm, a);
    }
    if (a.bulk_epilogue)
      return launch_pdl(wkv_gemm_pair_kernel<true, false>, grid, dim3(kGemmThreads), PairCfg::kSmemBytes, stream, 2,
                        tmA, tmW, xm, a);
    return launch_pdl(wkv_gemm_pair_kernel<false, false>, grid, dim3(kGemmThreads), PairCfg::kSmemBytes, stream, 2,
                      tmA, tmW, xm, a);
  }
  const int ar = gemm_a_rows(a.M);
  CUtensorMap tmA;
  const bool mapped =
      a.fp8 ? make_tmap_u8(&tmA, rows, static_cast<uint64_t>(a.M), static_cast<uint64_t>(a.K), static_cast<uint32_t>(ar))
            : make_tmap_bf16(&tmA, rows, static_cast<uint64_t>(a.M), static_cast<uint64_t>(a.K),
                             static_cast<uint32_t>(ar));
  if (!mapped) return cudaErrorInvalidValue;
  if (ar == 32) return launch_variant<32, 5>(tmA, tmB, a, ctas, stream);
  if (ar == 64) return launch_variant<64, 5>(tmA, tmB, a, ctas, stream);
  return launch_variant<128, 4>(tmA, tmB, a, ctas, stream);
}

}  // namespace engram
