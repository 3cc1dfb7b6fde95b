// Launchers shared by the translation units of libengram.so.  Host code only
// sees these declarations; each launcher queues its kernel on `stream` and
// returns the cudaError_t of the launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace engram {

// Launches `kernel` on `stream` with programmatic dependent launch allowed (the
// kernel may start while the previous kernel in the stream finishes; every
// kernel here calls griddepcontrol.wait before it touches memory an earlier
// kernel may still write, and triggers its dependents only after that wait)
// and, when cluster_x > 1, in clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Whether kernels on `device` can read p at address p: memory of that device,
// managed memory, or pinned host memory mapped at the same address.  Host code
// only; it allocates nothing and queues nothing.  A pointer that fails it
// (pageable host memory, another device's memory) would make the first kernel
// that dereferences it fault.
inline bool device_readable(const void* p, int device) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  switch (at.type) {
    case cudaMemoryTypeDevice: return at.device == device;
    case cudaMemoryTypeManaged: return true;
    case cudaMemoryTypeHost: return at.devicePointer == p;
    default: return false;
  }
}

// ---- rows: gather + dequantise (steps a1-a3) ------------------------------
struct GatherArgs {
  const int64_t* ids;       // [rows_total] global row ids (rows_total = M * n_cols)
  const uint8_t* table;     // [R, head_dim] e4m3 codes
  const void* scale;        // [R, head_dim/scale_block] fp32 or e8m0
  uint16_t* out;            // [rows_total, head_dim] bf16
  int64_t rows_total;
  int64_t R;                // rows of the table (of the shard)
  int64_t row0;             // global id of its first row: id i reads row i - row0
  int32_t head_dim;
  int32_t scale_block;
  int32_t scale_fmt;
  int32_t check_ids;
  unsigned long long* err;  // [0]: flags, [1]: count of ids out of range
  uint32_t* zero;           // words the kernel that follows needs cleared (may be null)
  int32_t n_zero;
};
cudaError_t launch_gather(const GatherArgs& a, int num_sms, cudaStream_t stream);
// MXFP8 operands for the block-scaled projection: the rows' e4m3 codes copied
// to codes [M, K] (a zero row for an id outside [0, R)) and their E8M0 scales
// (scale_block 32) to sfa in the projection's A-scale order: 512 bytes per
// (M tile of 128, K block of 128) at byte (m_tile * K/128 + k_block) * 512,
// byte 16*l + 4*q + j = scale of K-block j (of 32) of row l + 32*q of the tile
// (127, i.e. 1.0, for a zero row).  Uses ids, table, scale, rows_total, R,
// head_dim, check_ids, err, zero/n_zero of `a`.
cudaError_t launch_gather_codes(const GatherArgs& a, int n_cols, uint8_t* codes, uint8_t* sfa, int num_sms,
                                cudaStream_t stream);

// ---- projection (step a4) --------------------------------------------------
constexpr int kBM = 128;     // tokens per tile (MMA M)
constexpr int kBN = 256;     // kv columns per tile (MMA N)
constexpr int kBK = 64;      // K elements per pipeline stage (one 128-byte swizzle row)
constexpr int kGemmThreads = 192;

enum GemmOut : int32_t { kOutBf16 = 0, kOutPartial = 1, kOutFused = 2 };

struct GemmArgs {
  int64_t M;
  int32_t N;
  int32_t K;
  int32_t splits;        // split-K factor; K/kBK divisible by it
  int32_t kb_per_split;  // (K/kBK) / splits
  int32_t m_tiles;
  int32_t n_tiles;
  int32_t group_m;       // m-tiles per rasterisation group
  int64_t units;         // full_units + rem_tiles * rem_splits
  // Remainder split (splits == 1 only): the last rem_tiles tiles of the raster
  // order, which would otherwise fill only part of a last wave, are cut into
  // rem_splits K ranges of rem_kb K-blocks; each range stores its fp32 sums in
  // rem_ws and launch_reduce_remainder adds them up in range order into kv.
  int64_t full_units;
  int32_t rem_tiles;
  int32_t rem_splits;
  int32_t rem_kb;
  float* rem_ws;         // [rem_tiles * rem_splits, 128, 256]
  int32_t pair;          // CTA pairs (tcgen05 cta_group::2): units are 256 x 256 tiles, group_m counts M
                         // pairs; bf16 kv, whole K, launched in clusters of two
  int32_t out_mode;      // GemmOut
  int32_t bulk_epilogue; // plain epilogue stores by per-row bulk copies (large batches)
  int32_t keep_weight;   // weight tiles L2 evict-last (shared by many M tiles) instead of evict-first
  const uint8_t* wpack;  // the weight in tile-packed order (pack_wkv), or nullptr: read through tmB
  int32_t fp8;           // MXFP8 operands: A = table codes [M, K] u8, B = packed weight codes
  const uint8_t* sfa;    // fp8: A scales, [m_tiles, K/128, 512] (gather_codes layout)
  const uint8_t* sfb;    // fp8: B scales, [n_tiles, K/128, 1024] (pack_sfb layout)
  uint16_t* kv;          // kOutBf16: [M, N]
  float* part;           // kOutPartial: [splits, M, N]
  unsigned long long* err;
  // kOutFused (splits == 1): the gate and the residual add run in the epilogue
  const uint16_t* x;     // [M, hc, dim]
  const uint8_t* mask;   // [M] or nullptr
  const float* wprod;    // [hc, dim]
  uint16_t* out;         // [M, hc, dim]
  float* gsum;           // [M, hc, dim/256, 4]: block sums of h^2, key^2, h*w*key
  float* gates;          // [M, 4] the gates of every row, formed by the last key warp of its quarter
  uint32_t* counters;    // [m_tiles, 8]: key tiles done per lane quarter, then gates-ready flags; zeroed by the gather
  uint32_t* tickets;     // [2]: the next unit to take, CTAs finished; 0 between launches (the last CTA resets them)
  int32_t key_n_tiles;   // n-tiles of the keys (hc*dim/256); an M tile's key units precede its value units
  int32_t hold_ready_flags;  // test hook (engram_test_hook): never raise the gates-ready flags
  int32_t dim;
  int32_t hc;
  float eps;
  float clamp;
  float inv_sqrt_dim;
};
cudaError_t gemm_prepare();   // per-device one-time kernel attributes
// How many CTA pairs of the pair projection fit on the device at once (0: none).
int gemm_pair_slots(int num_sms);
// Rows of the A (gathered rows) box the projection uses for a batch of M tokens.
int gemm_a_rows(int64_t M);
// Whether the projection variant for M tokens has shared memory for the fused epilogue.
bool gemm_can_fuse(int64_t M);
// bf16 [rows, cols] row-major matrix, box = [box_rows, 64 columns], 128-byte swizzle.
bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);
// rows: the gathered rows [M, K], bf16 or (fp8) e4m3 codes (its tensor map is
// built here, to match the kernel variant); tmB: the weight's map, box [256
// rows, 64 columns] (unused when a.wpack is set).
cudaError_t launch_gemm(const void* rows, const CUtensorMap& tmB, const GemmArgs& a, int ctas,
                        cudaStream_t stream);
// The weight [N, K] (N a multiple of 256, K of 64) rewritten as 32 KB tiles,
// tile (n_tile, k_block) at byte offset (n_tile * K/64 + k_block) * 32768, each
// holding rows n_tile*256 .. +255, columns k_block*64 .. +63 exactly as a
// 128-byte-swizzled tensor copy of that box lands in shared memory.  `packed`
// holds N*K*2 bytes, 16-byte aligned.
cudaError_t launch_pack_wkv(const uint16_t* wkv, int64_t N, int64_t K, uint8_t* packed, cudaStream_t stream);
// The MXFP8 weight's E8M0 scales [N, K/32] in the projection's order: 1 KB per
// (n_tile, k_block of 128) at byte (n_tile * K/128 + k_block) * 1024; rows
// 0-127 of the tile in the first 512 bytes, 128-255 in the second; in each,
// byte 16*l + 4*q + j = scale of K-block j (of 32) of row l + 32*q.  The
// codes themselves are packed by launch_pack_wkv viewing [N, K] bytes as
// [N, K/2] 16-bit elements.
// kv of the remainder tiles from the workspace (after the projection, PDL).
cudaError_t launch_reduce_remainder(const GemmArgs& a, int num_sms, cudaStream_t stream);
cudaError_t launch_pack_sfb(const uint8_t* wkv_scale, int64_t N, int64_t K, uint8_t* packed, cudaStream_t stream);

// ---- gate and residual (steps a5-a8) ---------------------------------------
struct GateArgs {
  const uint16_t* kv;     // [M, N] bf16 (when part == nullptr)
  const float* part;      // [splits, M, N] fp32 partial sums of kv, or nullptr
  int32_t splits;
  const uint16_t* x;      // [M, hc, dim]
  const uint8_t* mask;    // [M] or nullptr
  const float* wprod;     // [hc, dim] q_weight * k_weight
  uint16_t* out;          // [M, hc, dim]
  float* gates;           // [M, hc] or nullptr
  int64_t M;
  int32_t dim;
  int32_t hc;
  float eps;
  float clamp;
  float inv_sqrt_dim;
  int32_t cluster;        // CTAs per token (set by launch_gate)
  unsigned long long* err;  // device error word (bounded waits), or nullptr
  int32_t num_sms;        // SMs of the device (0: unknown)
  int32_t wprod_after_wait;  // wprod is written by a kernel of the same call: read it after the
                             // dependency wait (otherwise it is read before, to hide its latency)
};
cudaError_t gate_prepare();   // per-device one-time kernel attributes
cudaError_t launch_gate(const GateArgs& a, cudaStream_t stream);

// kv[m, n] = bf16(sum over splits, in order, of part[s, m, n])
cudaError_t launch_reduce_partials(const float* part, int32_t splits, int64_t M, int32_t N, uint16_t* kv,
                                   int num_sms, cudaStream_t stream);

// wprod[i] = fp32(q[i]) * fp32(k[i])
cudaError_t launch_weight_product(const uint16_t* q, const uint16_t* k, float* wprod, int64_t n,
                                  cudaStream_t stream);

}  // namespace engram
