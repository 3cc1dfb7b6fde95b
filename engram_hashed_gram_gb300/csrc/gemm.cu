// Step a4 of the Engram layer, the wkv projection (atlas.klimoza.dev
// "deepseek-v4.1 / engram-second", `Engram.forward`:
// kv = wkv(embed(hash_ids).flatten(-2))): kv[m, n] = sum_k E[m, k] * W[n, k],
// E the gathered bf16 rows [M, K], W the Linear's [N, K] bf16 weight, fp32
// accumulation.
//
// Design (sm_103a, one CTA per SM, persistent):
//  * a work unit is a 128 x 256 output tile restricted to one K range
//    (split-K); units are dealt round-robin to the CTAs;
//  * warp 0 (one thread) streams A = E[A_ROWS rows, 64 k] and B = W[256 rows,
//    64 k] boxes with TMA (128-byte swizzle) into a STAGES-deep shared-memory
//    ring;
//  * warp 1 (one thread) issues tcgen05.mma (M=128, N=256, K=16, bf16 -> fp32)
//    into one of two 256-column tensor-memory accumulators and commits each
//    stage back to the producer;
//  * warps 2-5 drain the other accumulator with tcgen05.ld and write either the
//    bf16 kv (round to nearest even) or the fp32 partial sums of a K range;
//  * no cluster, no multicast: the L2 serves the reuse of E and W across CTAs.
// Variants: A_ROWS = 128 with 4 stages in general; for batches of at most 64
// or 32 tokens the A box holds only 64 or 32 rows, and the shared memory that
// frees goes to a deeper ring (5 or 6 stages), i.e. more of the weight stream
// in flight per SM.  The MMA still reads 128 rows of A: rows past the box are
// whatever the neighbouring shared memory holds, their accumulator rows are
// never stored, and a row of D depends on its own row of A only.  Rows of the
// last M tile past M read as zeros (TMA bounds fill) and are not stored.
#include <mutex>

#include "common.cuh"
#include "internal.cuh"

namespace engram {
namespace {

constexpr int kBBytes = kBN * kBK * 2;        // 32 KB
constexpr uint32_t kTmemCols = 2 * kBN;        // two fp32 accumulators

template <int A_ROWS, int STAGES>
struct Cfg {
  static constexpr int kABytes = A_ROWS * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarOffset = STAGES * kStageBytes;
  static constexpr int kNumBars = 2 * STAGES + 2 + 2 + 1;
  static constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + kBarOffset + kNumBars * 8 + 16;
  static_assert(kABytes % 1024 == 0, "A stages must stay 1024-byte aligned");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

__device__ __forceinline__ void unit_coords(const GemmArgs& a, int64_t u, int& mt, int& nt, int& sp) {
  sp = static_cast<int>(u % a.splits);
  const int64_t t = u / a.splits;
  const int64_t group_tiles = static_cast<int64_t>(a.group_m) * a.n_tiles;
  const int64_t g = t / group_tiles;
  const int64_t r = t - g * group_tiles;
  const int gm0 = static_cast<int>(g) * a.group_m;
  const int gm = min(a.group_m, a.m_tiles - gm0);
  nt = static_cast<int>(r / gm);
  mt = gm0 + static_cast<int>(r % gm);
}

__device__ __forceinline__ void raise_abort(volatile int* abort_flag, unsigned long long* err) {
  *abort_flag = 1;
  atomicOr(err, kErrTimeout);
}

template <int A_ROWS, int STAGES>
__global__ void __launch_bounds__(kGemmThreads, 1)
    wkv_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmArgs a) {
  using C = Cfg<A_ROWS, STAGES>;
  constexpr int kStages = STAGES;
  constexpr int kABytes = C::kABytes;
  constexpr int kStageBytes = C::kStageBytes;
  constexpr int kBarOffset = C::kBarOffset;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smem + kStages * kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOffset);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

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
      const uint64_t pol_w = policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued[kStages] = {};
      bool ok = true;
      // The weight does not depend on the kernel queued before this one (the
      // gather): the first stages of the first unit get their weight tile while
      // the gathered rows are still being written.
      int pre = 0;
      if (static_cast<int64_t>(blockIdx.x) < a.units) {
        int mt, nt, sp;
        unit_coords(a, blockIdx.x, mt, nt, sp);
        pre = min(kStages, a.kb_per_split);
        for (int i = 0; i < pre; ++i) {   // fresh ring: every stage is free
          mbar_arrive_expect_tx(&full[i], kStageBytes);
          tma_load_2d_hint(smB + i * kBBytes, &tmB, &full[i], (sp * a.kb_per_split + i) * kBK, nt * kBN, pol_w);
        }
      }
      grid_dependency_wait();     // the gathered rows are written by the gather kernel
      for (int64_t u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
        // the kernel queued after this one (the gate) may start arriving once
        // every CTA has begun its last unit
        if (u + gridDim.x >= a.units) grid_launch_dependents();
        int mt, nt, sp;
        unit_coords(a, u, mt, nt, sp);
        const int kb0 = sp * a.kb_per_split;
        for (int kb = 0; kb < a.kb_per_split; ++kb) {
          if (u == blockIdx.x && kb < pre) {
            // weight tile already in flight on this stage: add the rows
            tma_load_2d(smA + stage * kABytes, &tmA, &full[stage], (kb0 + kb) * kBK, mt * kBM);
          } else {
            if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[stage], kStageBytes);
            tma_load_2d(smA + stage * kABytes, &tmA, &full[stage], (kb0 + kb) * kBK, mt * kBM);
            tma_load_2d_hint(smB + stage * kBBytes, &tmB, &full[stage], (kb0 + kb) * kBK, nt * kBN, pol_w);
          }
          ++issued[stage];
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
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
      for (int64_t u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
        if (u + gridDim.x >= a.units) grid_launch_dependents();
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        for (int kb = 0; kb < a.kb_per_split; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(smA + stage * kABytes));
          const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(smB + stage * kBBytes));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // +32 bytes per K step of 16 bf16 = +2 in the start-address field
            umma_bf16(d_tmem, adesc + 2ull * kk, bdesc + 2ull * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
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
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int64_t u = blockIdx.x; u < a.units; u += gridDim.x) {
      if (u + gridDim.x >= a.units) grid_launch_dependents();
      int mt, nt, sp;
      unit_coords(a, u, mt, nt, sp);
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int64_t m = static_cast<int64_t>(mt) * kBM + q * 32 + lane;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kBN);
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), r);
        tmem_ld_wait();
        if (m < a.M) {
          const int n0 = nt * kBN + c * 32;
          if (a.out_mode == kOutBf16) {
            uint4* dst = reinterpret_cast<uint4*>(a.kv + m * a.N + n0);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              dst[j] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * j + 0]), __uint_as_float(r[8 * j + 1])),
                                  pack_bf16x2(__uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3])),
                                  pack_bf16x2(__uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5])),
                                  pack_bf16x2(__uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7])));
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(a.part + (static_cast<int64_t>(sp) * a.M + m) * a.N + n0);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              dst[j] = make_float4(__uint_as_float(r[4 * j + 0]), __uint_as_float(r[4 * j + 1]),
                                   __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok && lane == 0) raise_abort(abort_flag, a.err);
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

template <int A_ROWS, int STAGES>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(wkv_gemm_kernel<A_ROWS, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(Cfg<A_ROWS, STAGES>::kSmemBytes));
}

template <int A_ROWS, int STAGES>
cudaError_t launch_variant(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a, int ctas,
                           cudaStream_t stream) {
  return launch_pdl(wkv_gemm_kernel<A_ROWS, STAGES>, dim3(static_cast<unsigned>(ctas)), dim3(kGemmThreads),
                    Cfg<A_ROWS, STAGES>::kSmemBytes, stream, 1, tmA, tmB, a);
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

cudaError_t gemm_prepare() {
  cudaError_t e = set_smem_attr<128, 4>();
  if (e == cudaSuccess) e = set_smem_attr<64, 5>();
  if (e == cudaSuccess) e = set_smem_attr<32, 6>();
  return e;
}

cudaError_t launch_gemm(const uint16_t* rows, const CUtensorMap& tmB, const GemmArgs& a, int ctas,
                        cudaStream_t stream) {
  if (a.units == 0) return cudaSuccess;
  const int ar = gemm_a_rows(a.M);
  CUtensorMap tmA;
  if (!make_tmap_bf16(&tmA, rows, static_cast<uint64_t>(a.M), static_cast<uint64_t>(a.K), static_cast<uint32_t>(ar)))
    return cudaErrorInvalidValue;
  if (ar == 32) return launch_variant<32, 6>(tmA, tmB, a, ctas, stream);
  if (ar == 64) return launch_variant<64, 5>(tmA, tmB, a, ctas, stream);
  return launch_variant<128, 4>(tmA, tmB, a, ctas, stream);
}

}  // namespace engram
