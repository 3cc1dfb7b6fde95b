// Launchers shared by the translation units of libengram.so.  Host code only
// sees these declarations; each launcher queues its kernel on `stream` and
// returns the cudaError_t of the launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace engram {

// ---- rows: gather + dequantise (steps a1-a3) ------------------------------
struct GatherArgs {
  const int64_t* ids;       // [rows_total] global row ids (rows_total = M * n_cols)
  const uint8_t* table;     // [R, head_dim] e4m3 codes
  const void* scale;        // [R, head_dim/scale_block] fp32 or e8m0
  uint16_t* out;            // [rows_total, head_dim] bf16
  int64_t rows_total;
  int64_t R;
  int32_t head_dim;
  int32_t scale_block;
  int32_t scale_fmt;
  int32_t check_ids;
  unsigned long long* err;  // [0]: flags, [1]: count of ids out of range
};
cudaError_t launch_gather(const GatherArgs& a, int num_sms, cudaStream_t stream);

// ---- projection (step a4) --------------------------------------------------
constexpr int kBM = 128;     // tokens per tile (MMA M)
constexpr int kBN = 256;     // kv columns per tile (MMA N)
constexpr int kBK = 64;      // K elements per pipeline stage (one 128-byte swizzle row)
constexpr int kStages = 4;
constexpr int kGemmThreads = 192;

enum GemmOut : int32_t { kOutBf16 = 0, kOutPartial = 1 };

struct GemmArgs {
  int64_t M;
  int32_t N;
  int32_t K;
  int32_t splits;        // split-K factor; K/kBK divisible by it
  int32_t kb_per_split;  // (K/kBK) / splits
  int32_t m_tiles;
  int32_t n_tiles;
  int32_t group_m;       // m-tiles per rasterisation group
  int64_t units;         // m_tiles * n_tiles * splits
  int32_t out_mode;      // GemmOut
  uint16_t* kv;          // kOutBf16: [M, N]
  float* part;           // kOutPartial: [splits, M, N]
  unsigned long long* err;
};
size_t gemm_smem_bytes();
cudaError_t gemm_prepare();   // per-device one-time kernel attributes
cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a, int ctas,
                        cudaStream_t stream);

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
};
cudaError_t launch_gate(const GateArgs& a, cudaStream_t stream);

// kv[m, n] = bf16(sum over splits, in order, of part[s, m, n])
cudaError_t launch_reduce_partials(const float* part, int32_t splits, int64_t M, int32_t N, uint16_t* kv,
                                   int num_sms, cudaStream_t stream);

// wprod[i] = fp32(q[i]) * fp32(k[i])
cudaError_t launch_weight_product(const uint16_t* q, const uint16_t* k, float* wprod, int64_t n,
                                  cudaStream_t stream);

}  // namespace engram
