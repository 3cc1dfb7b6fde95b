// Steps a1-a3 of the Engram layer: id range check, row gather and
// dequantisation (atlas.klimoza.dev "deepseek-v4.1 / engram-second",
// `ParallelEngramEmbedding.forward`): for row r = ids[i] - row0 (row0: the
// global id of the table's first row, non-zero for one shard of a row-split
// table),
//   out[i, f] = bf16_rn( fp32(e4m3 code[r, f]) *_rn scale[r, f / scale_block] )
// and a zero row when r is outside [0, R).  The difference is taken in
// unsigned 64-bit arithmetic, so every id below row0 (however negative) wraps
// past R and is outside too.
//
// One thread owns one 16-byte chunk of a row (16 codes): consecutive threads
// read consecutive chunks of the same 256-byte row, so each row is one fully
// used set of 32-byte sectors, and write 32 bytes of bf16 each.  The table is
// read once with no L1 allocation.  The fp8 -> half conversion is exact and the
// product is a single fp32 multiply (no FMA contraction), so the result is
// bit-identical to the definition.
//
// gather_codes_kernel serves the MXFP8 weight: it copies the codes unchanged
// and places the E8M0 scales in the block-scaled projection's order.
#include "common.cuh"
#include "internal.cuh"

namespace engram {
namespace {

__device__ __forceinline__ uint4 ld_stream_v4(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float e8m0_to_float(uint32_t e) {
  if (e == 0u) return __uint_as_float(0x00400000u);   // 2^-127, an fp32 subnormal
  if (e == 255u) return __uint_as_float(0x7FC00000u);
  return __uint_as_float(e << 23);
}

// 4 codes (one 32-bit word, lowest byte first) -> 4 bf16 in two words
__device__ __forceinline__ void dequant4(uint32_t w, float s, uint32_t& o0, uint32_t& o1) {
  const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xFFFFu), __NV_E4M3);
  const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
  const float2 f01 = __half22float2(__half2(h01));
  const float2 f23 = __half22float2(__half2(h23));
  o0 = pack_bf16x2(__fmul_rn(f01.x, s), __fmul_rn(f01.y, s));
  o1 = pack_bf16x2(__fmul_rn(f23.x, s), __fmul_rn(f23.y, s));
}

// SHIFT: head_dim / 16 and scale_block are powers of two (cpr_log2,
// sb_log2), and the chunk count fits 32 bits: the index arithmetic is shifts
// and 32-bit adds instead of 64-bit divisions, which took half the kernel's
// issue slots.
template <int SCALE_FMT, bool SHIFT>
__global__ void __launch_bounds__(256) gather_dequant_kernel(GatherArgs a, int cpr_log2, int sb_log2) {
  grid_dependency_wait();        // the ids may come from the previous kernel
  grid_launch_dependents();      // let the projection start its weight stream
  if (a.zero != nullptr) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.n_zero; i += gridDim.x * blockDim.x) a.zero[i] = 0u;
  }
  const int cpr = a.head_dim >> 4;              // 16-byte chunks per row
  const int nb = a.head_dim / a.scale_block;
  const int64_t total = a.rows_total * cpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    int64_t row;
    int ch;
    if (SHIFT) {
      const uint32_t i32 = static_cast<uint32_t>(i);
      row = static_cast<int64_t>(i32 >> cpr_log2);
      ch = static_cast<int>(i32 & ((1u << cpr_log2) - 1u));
    } else {
      row = i / cpr;
      ch = static_cast<int>(i - row * cpr);
    }
    const uint64_t ur = static_cast<uint64_t>(__ldg(a.ids + row)) - static_cast<uint64_t>(a.row0);
    const int64_t r = static_cast<int64_t>(ur);
    uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = make_uint4(0u, 0u, 0u, 0u);
    if (ur < static_cast<uint64_t>(a.R)) {
      const uint4 c = ld_stream_v4(a.table + r * a.head_dim + ch * 16);
      const int blk = SHIFT ? (ch * 16) >> sb_log2 : (ch * 16) / a.scale_block;
      float s;
      if (SCALE_FMT == 0) {
        s = __ldg(static_cast<const float*>(a.scale) + r * nb + blk);
      } else {
        s = e8m0_to_float(__ldg(static_cast<const uint8_t*>(a.scale) + r * nb + blk));
      }
      dequant4(c.x, s, lo.x, lo.y);
      dequant4(c.y, s, lo.z, lo.w);
      dequant4(c.z, s, hi.x, hi.y);
      dequant4(c.w, s, hi.z, hi.w);
    } else if (a.check_ids && ch == 0) {
      atomicAdd(a.err + 1, 1ull);
      atomicOr(a.err, kErrRange);
    }
    uint4* dst = reinterpret_cast<uint4*>(a.out + row * a.head_dim + ch * 16);
    dst[0] = lo;
    dst[1] = hi;
  }
}

// One thread per 16-byte chunk of a row's codes; the first head_dim/32
// threads of a row also place its scales.
__global__ void __launch_bounds__(256) gather_codes_kernel(GatherArgs a, int n_cols, int64_t kbt,
                                                           uint8_t* __restrict__ codes, uint8_t* __restrict__ sfa) {
  grid_dependency_wait();        // the ids may come from the previous kernel
  grid_launch_dependents();      // let the projection start its weight stream
  if (a.zero != nullptr) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.n_zero; i += gridDim.x * blockDim.x) a.zero[i] = 0u;
  }
  const int cpr = a.head_dim >> 4;
  const int nb = a.head_dim >> 5;
  const int64_t K = static_cast<int64_t>(n_cols) * a.head_dim;
  const int64_t total = a.rows_total * cpr;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t row = i / cpr;
    const int ch = static_cast<int>(i - row * cpr);
    const int64_t m = row / n_cols;
    const int c = static_cast<int>(row - m * n_cols);
    const uint64_t ur = static_cast<uint64_t>(__ldg(a.ids + row)) - static_cast<uint64_t>(a.row0);
    const int64_t r = static_cast<int64_t>(ur);
    const bool valid = ur < static_cast<uint64_t>(a.R);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (valid) {
      v = ld_stream_v4(a.table + r * a.head_dim + ch * 16);
    } else if (a.check_ids && ch == 0) {
      atomicAdd(a.err + 1, 1ull);
      atomicOr(a.err, kErrRange);
    }
    *reinterpret_cast<uint4*>(codes + m * K + static_cast<int64_t>(c) * a.head_dim + ch * 16) = v;
    if (ch < nb) {
      const uint8_t sc = valid ? __ldg(static_cast<const uint8_t*>(a.scale) + r * nb + ch) : uint8_t{127};
      const int64_t q = (static_cast<int64_t>(c) * a.head_dim >> 5) + ch;   // K-block of 32
      const int t = static_cast<int>(m & 127);
      sfa[(((m >> 7) * kbt + (q >> 2)) << 9) + ((t & 31) << 4) + ((t >> 5) << 2) + (q & 3)] = sc;
    }
  }
}

}  // namespace

cudaError_t launch_gather_codes(const GatherArgs& a, int n_cols, uint8_t* codes, uint8_t* sfa, int num_sms,
                                cudaStream_t stream) {
  const int64_t total = a.rows_total * (a.head_dim >> 4);
  if (total == 0) return cudaSuccess;
  const int64_t K = static_cast<int64_t>(n_cols) * a.head_dim;
  if (K % 128 != 0 || a.head_dim % 32 != 0) return cudaErrorInvalidValue;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  return launch_pdl(gather_codes_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, 1, a, n_cols,
                    K / 128, codes, sfa);
}

cudaError_t launch_gather(const GatherArgs& a, int num_sms, cudaStream_t stream) {
  const int64_t total = a.rows_total * (a.head_dim >> 4);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;   // 8 resident CTAs of 256 per SM
  if (blocks > cap) blocks = cap;
  const dim3 grid(static_cast<unsigned>(blocks));
  const int cpr = a.head_dim >> 4;
  const int cl = __builtin_ctz(static_cast<unsigned>(cpr));
  const int sl = __builtin_ctz(static_cast<unsigned>(a.scale_block));
  const bool shift = (1 << cl) == cpr && (1 << sl) == a.scale_block && total + static_cast<int64_t>(blocks) * threads <
                                                                           (int64_t{1} << 32);
  if (shift) {
    if (a.scale_fmt == 0) return launch_pdl(gather_dequant_kernel<0, true>, grid, dim3(threads), 0, stream, 1, a, cl, sl);
    return launch_pdl(gather_dequant_kernel<1, true>, grid, dim3(threads), 0, stream, 1, a, cl, sl);
  }
  if (a.scale_fmt == 0) return launch_pdl(gather_dequant_kernel<0, false>, grid, dim3(threads), 0, stream, 1, a, 0, 0);
  return launch_pdl(gather_dequant_kernel<1, false>, grid, dim3(threads), 0, stream, 1, a, 0, 0);
}

}  // namespace engram
