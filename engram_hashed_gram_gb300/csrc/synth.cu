// Device twin of the seeded table generator (include/engram_synth.h).  Input
// generation for tests and benchmarks only: it writes exactly what
// engram_hashed_gram_gb300/synth.py's table_rows() computes on the host.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/engram_synth.h"

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t draw(uint64_t key, uint64_t counter) {
  return mix64(key + (counter + 1ull) * kGamma);
}

// The 64 KB code quantile table is staged in shared memory.
__global__ void __launch_bounds__(512) fill_codes_kernel(uint8_t* __restrict__ table, int64_t row_begin,
                                                         int64_t row_end, int head_dim, uint64_t key,
                                                         const uint8_t* __restrict__ qtable) {
  extern __shared__ uint4 s_q4[];
  const uint4* q4 = reinterpret_cast<const uint4*>(qtable);
  for (int i = threadIdx.x; i < 65536 / 16; i += blockDim.x) s_q4[i] = q4[i];
  __syncthreads();
  const uint8_t* sq = reinterpret_cast<const uint8_t*>(s_q4);
  const int cpr = head_dim / 16;
  const int words = head_dim / 4;
  const int64_t total = (row_end - row_begin) * cpr;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = row_begin + i / cpr;
    const int ch = static_cast<int>(i % cpr);
    const uint64_t c0 = static_cast<uint64_t>(row) * words + static_cast<uint64_t>(ch) * 4;
    uint32_t out[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint64_t d = draw(key, c0 + w);
      out[w] = static_cast<uint32_t>(sq[d & 0xFFFF]) | (static_cast<uint32_t>(sq[(d >> 16) & 0xFFFF]) << 8) |
               (static_cast<uint32_t>(sq[(d >> 32) & 0xFFFF]) << 16) |
               (static_cast<uint32_t>(sq[(d >> 48) & 0xFFFF]) << 24);
    }
    *reinterpret_cast<uint4*>(table + row * head_dim + ch * 16) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

__global__ void fill_scales_kernel(float* __restrict__ scale, int64_t row_begin, int64_t row_end, int nb,
                                   uint64_t key, const float* __restrict__ qtable) {
  const int64_t total = (row_end - row_begin) * nb;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint64_t c = static_cast<uint64_t>(row_begin) * nb + static_cast<uint64_t>(i);
    scale[c] = __ldg(qtable + (draw(key, c) >> 48));
  }
}

__global__ void fill_scales_e8m0_kernel(uint8_t* __restrict__ scale, int64_t row_begin, int64_t row_end, int nb,
                                        uint64_t key, const uint8_t* __restrict__ qtable) {
  const int64_t total = (row_end - row_begin) * nb;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint64_t c = static_cast<uint64_t>(row_begin) * nb + static_cast<uint64_t>(i);
    scale[c] = __ldg(qtable + (draw(key, c) >> 48));
  }
}

}  // namespace

extern "C" int32_t engram_synth_fill_scales_e8m0(uint8_t* scale, int64_t row_begin, int64_t row_end,
                                                 int32_t head_dim, int32_t scale_block, uint64_t key_scales,
                                                 const uint8_t* e8m0_qtable, engram_synth_stream_t stream) {
  if (scale == nullptr || e8m0_qtable == nullptr || row_begin < 0 || row_end < row_begin || head_dim <= 0 ||
      scale_block <= 0 || head_dim % scale_block != 0)
    return -1;
  if (row_end == row_begin) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -3;
  fill_scales_e8m0_kernel<<<sms * 4, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      scale, row_begin, row_end, head_dim / scale_block, key_scales, e8m0_qtable);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

extern "C" int32_t engram_synth_fill_table(uint8_t* table, float* scale, int64_t row_begin, int64_t row_end,
                                           int32_t head_dim, int32_t scale_block, uint64_t key_codes,
                                           uint64_t key_scales, const uint8_t* code_qtable,
                                           const float* scale_qtable, engram_synth_stream_t stream) {
  if (table == nullptr || code_qtable == nullptr || row_begin < 0 || row_end < row_begin || head_dim <= 0 ||
      head_dim % 16 != 0 || scale_block <= 0 || head_dim % scale_block != 0 ||
      (reinterpret_cast<uintptr_t>(table) & 15) != 0 || (reinterpret_cast<uintptr_t>(code_qtable) & 15) != 0)
    return -1;
  if (scale != nullptr && scale_qtable == nullptr) return -1;
  if (row_end == row_begin) return 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -3;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(fill_codes_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 65536) != cudaSuccess)
      return -3;
    attr_done = true;
  }
  fill_codes_kernel<<<sms * 2, 512, 65536, s>>>(table, row_begin, row_end, head_dim, key_codes, code_qtable);
  if (cudaGetLastError() != cudaSuccess) return -3;
  if (scale != nullptr) {
    fill_scales_kernel<<<sms * 4, 256, 0, s>>>(scale, row_begin, row_end, head_dim / scale_block, key_scales,
                                               scale_qtable);
    if (cudaGetLastError() != cudaSuccess) return -3;
  }
  return 0;
}
