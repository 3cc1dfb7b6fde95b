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
#include <cstdlib>
#include <cstring>

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

template <int SCALE_FMT>
__global__ void __launch_bounds__(256) gather_dequant_kernel(GatherArgs a) {
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
    const int64_t row = i / cpr;
    const int ch = static_cast<int>(i - row * cpr);
    const uint64_t ur = static_cast<uint64_t>(__ldg(a.ids + row)) - static_cast<uint64_t>(a.row0);
    const int64_t r = static_cast<int64_t>(ur);
    uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = make_uint4(0u, 0u, 0u, 0u);
    if (ur < static_cast<uint64_t>(a.R)) {
      const uint4 c = ld_stream_v4(a.table + r * a.head_dim + ch * 16);
      const int blk = (ch * 16) / a.scale_block;
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

// ---------------------------------------------------------------- staged gather
// The same rows and bits as gather_dequant_kernel, with the table rows staged
// through shared memory by the copy engine.  Each warp takes batches of 32
// rows: lane l reads the id of row l of the batch (one coalesced load for the
// warp), issues one bulk copy (cp.async.bulk) of that row's codes into the
// warp's slot -- all 32 copies counted on one mbarrier -- and loads the row's
// scales (at most 16 bytes) into registers.  While a batch is in flight the
// warp dequantises the previous one from shared memory (two slots per warp):
// lanes 16h..16h+15 cover one row's 16 chunks of 16 codes, taking the row's
// scales from its lane by shuffle, so each store instruction writes two whole
// bf16 rows.  No thread waits on a chain of dependent loads of its own, and an
// SM keeps up to 16 batches (128 KB of codes) in flight.  Used for a table in
// the device's own memory, head_dim <= 256, a 16-byte-aligned table and
// 4-byte scale words per row; other tables take gather_dequant_kernel.
constexpr int kStagedWarps = 8;
constexpr int kStagedSlotBytes = 32 * 256;
constexpr int kStagedSmem = kStagedWarps * 2 * kStagedSlotBytes + kStagedWarps * 2 * 8;

template <int SCALE_FMT>
__global__ void __launch_bounds__(kStagedWarps * 32, 1) gather_staged_kernel(GatherArgs a) {
  extern __shared__ __align__(128) uint8_t gsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* slots = gsm + warp * 2 * kStagedSlotBytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(gsm + kStagedWarps * 2 * kStagedSlotBytes) + warp * 2;
  if (lane == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbarrier_init();
  }
  __syncwarp();
  grid_dependency_wait();        // the ids may come from the previous kernel
  grid_launch_dependents();      // let the projection start its weight stream
  if (a.zero != nullptr) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.n_zero; i += gridDim.x * blockDim.x) a.zero[i] = 0u;
  }
  const int nb = a.head_dim / a.scale_block;
  const int swords = (nb * (SCALE_FMT == 0 ? 4 : 1)) >> 2;   // 32-bit scale words per row (1..4)
  const int cpr = a.head_dim >> 4;                           // 16-byte chunks per row
  const int64_t batches = (a.rows_total + 31) >> 5;
  const int64_t wstride = static_cast<int64_t>(gridDim.x) * kStagedWarps;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kStagedWarps + warp;
  const uint32_t* scale_words = static_cast<const uint32_t*>(a.scale);
  const uint64_t pol = policy_evict_first();

  // per slot (two named copies, so that they stay in registers): the rows of
  // the batch with an id inside the table, and lane l's scale words of row l
  uint32_t vmask0 = 0u, vmask1 = 0u;
  uint32_t sw0[4] = {0u, 0u, 0u, 0u}, sw1[4] = {0u, 0u, 0u, 0u};
  auto issue = [&](int64_t b, int slot) {
    const int64_t row = (b << 5) + lane;
    bool valid = false;
    uint64_t ur = 0;
    if (row < a.rows_total) {
      ur = static_cast<uint64_t>(__ldg(a.ids + row)) - static_cast<uint64_t>(a.row0);
      valid = ur < static_cast<uint64_t>(a.R);
      if (!valid && a.check_ids) {
        atomicAdd(a.err + 1, 1ull);
        atomicOr(a.err, kErrRange);
      }
    }
    const uint32_t vm = __ballot_sync(0xFFFFFFFFu, valid);
    if (slot) vmask1 = vm; else vmask0 = vm;
    const uint32_t total = static_cast<uint32_t>(__popc(vm)) * static_cast<uint32_t>(a.head_dim);
    if (lane == 0) mbar_arrive_expect_tx(&bar[slot], total);
    __syncwarp();
    if (valid) {
      bulk_load_hint(slots + slot * kStagedSlotBytes + lane * a.head_dim,
                     a.table + static_cast<int64_t>(ur) * a.head_dim, static_cast<uint32_t>(a.head_dim), &bar[slot],
                     pol);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t v = q < swords ? __ldg(scale_words + static_cast<int64_t>(ur) * swords + q) : 0u;
        if (slot) sw1[q] = v; else sw0[q] = v;
      }
    }
  };

  uint32_t phase[2] = {0u, 0u};
  uint32_t armed[2] = {0u, 0u};  // copies issued into each slot and not yet waited for
  bool ok = true;
  int slot = 0;
  if (first < batches) {
    issue(first, 0);
    armed[0] = 1u;
  }
  for (int64_t b = first; b < batches; b += wstride, slot ^= 1) {
    if (b + wstride < batches) {
      fence_proxy_async_shared();   // this warp's earlier reads of the slot precede the copies into it
      issue(b + wstride, slot ^ 1);
      armed[slot ^ 1] = 1u;
    }
    if (!mbar_wait(&bar[slot], phase[slot], nullptr)) {
      ok = false;
      break;
    }
    phase[slot] ^= 1u;
    armed[slot] = 0u;
    const uint8_t* base = slots + slot * kStagedSlotBytes;
    for (int j = 0; j < 32 * cpr; j += 32) {
      const int t = j + lane;
      const int r = t / cpr;                       // row of the batch
      const int ch = t - r * cpr;
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) w[q] = __shfl_sync(0xFFFFFFFFu, slot ? sw1[q] : sw0[q], r);
      const int64_t row = (b << 5) + r;
      if (row >= a.rows_total) continue;
      uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = make_uint4(0u, 0u, 0u, 0u);
      if ((((slot ? vmask1 : vmask0) >> r) & 1u) != 0u) {
        const uint4 c = ld_shared_v4(smem_u32(base + r * a.head_dim + ch * 16));
        const int blk = (ch * 16) / a.scale_block;
        float sc;
        if (SCALE_FMT == 0) {
          sc = __uint_as_float(blk == 0 ? w[0] : blk == 1 ? w[1] : blk == 2 ? w[2] : w[3]);
        } else {
          const uint32_t word = (blk >> 2) == 0 ? w[0] : (blk >> 2) == 1 ? w[1] : (blk >> 2) == 2 ? w[2] : w[3];
          sc = e8m0_to_float((word >> (8 * (blk & 3))) & 0xFFu);
        }
        dequant4(c.x, sc, lo.x, lo.y);
        dequant4(c.y, sc, lo.z, lo.w);
        dequant4(c.z, sc, hi.x, hi.y);
        dequant4(c.w, sc, hi.z, hi.w);
      }
      uint4* dst = reinterpret_cast<uint4*>(a.out + row * a.head_dim + ch * 16);
      dst[0] = lo;
      dst[1] = hi;
    }
    __syncwarp();                                   // the slot is free for the batch after next
  }
  if (!ok) {
    if (lane == 0) atomicOr(a.err, kErrTimeout);
    // let the copies in flight land before the CTA can exit
    for (int i = 0; i < 2; ++i)
      if (armed[i]) mbar_wait(&bar[i], phase[i], nullptr, kDrainLimitNs);
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

// The staged kernel unless ENGRAM_GATHER=plain (measurements).
bool staged_gather_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("ENGRAM_GATHER");
    return !(e != nullptr && std::strcmp(e, "plain") == 0);
  }();
  return on;
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

bool staged_gather_fits(const GatherArgs& a) {
  const int nb = a.head_dim / a.scale_block;
  const int sbytes = nb * (a.scale_fmt == 0 ? 4 : 1);
  return a.table_on_device && a.head_dim <= 256 && a.head_dim % 16 == 0 && sbytes % 4 == 0 && sbytes <= 16 &&
         (reinterpret_cast<uintptr_t>(a.table) & 15u) == 0 && (reinterpret_cast<uintptr_t>(a.scale) & 3u) == 0;
}

cudaError_t gather_prepare() {
  cudaError_t e = cudaFuncSetAttribute(gather_staged_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kStagedSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gather_staged_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kStagedSmem);
  return e;
}

cudaError_t launch_gather(const GatherArgs& a, int num_sms, cudaStream_t stream) {
  const int64_t total = a.rows_total * (a.head_dim >> 4);
  if (total == 0) return cudaSuccess;
  if (staged_gather_enabled() && staged_gather_fits(a)) {
    const int64_t batches = (a.rows_total + 31) / 32;
    int64_t blocks = (batches + kStagedWarps - 1) / kStagedWarps;
    if (blocks > num_sms) blocks = num_sms;
    const dim3 grid(static_cast<unsigned>(blocks));
    if (a.scale_fmt == 0)
      return launch_pdl(gather_staged_kernel<0>, grid, dim3(kStagedWarps * 32), kStagedSmem, stream, 1, a);
    return launch_pdl(gather_staged_kernel<1>, grid, dim3(kStagedWarps * 32), kStagedSmem, stream, 1, a);
  }
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;   // 8 resident CTAs of 256 per SM
  if (blocks > cap) blocks = cap;
  const dim3 grid(static_cast<unsigned>(blocks));
  if (a.scale_fmt == 0) return launch_pdl(gather_dequant_kernel<0>, grid, dim3(threads), 0, stream, 1, a);
  return launch_pdl(gather_dequant_kernel<1>, grid, dim3(threads), 0, stream, 1, a);
}

}  // namespace engram
