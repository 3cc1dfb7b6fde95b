// Steps a5-a8 of the Engram layer (atlas.klimoza.dev "deepseek-v4.1 /
// engram-second", `Engram.forward`; zhuai.tech "Engram in DeepSeek V4.1 Flash",
// section "Step 3: Inject memory at the correct layer boundary"):
//   key[s, d] = kv[s*dim + d], value[d] = kv[hc*dim + d]   (bf16)
//   rstd[s]   = 1/sqrt(mean_d h^2 + eps) * 1/sqrt(mean_d key^2 + eps)
//   dot[s]    = (sum_d h * (q_weight*k_weight) * key) * rstd * dim^-0.5
//   gate[s]   = sigmoid(copysign(sqrt(max(|dot|, clamp)), dot)), 0 if masked
//   out[s, d] = bf16(h + gate[s] * value[d]); masked tokens copy x bit-for-bit.
//
// A token is handled by a cluster of G CTAs (G = 4 for dim = 5120).  The
// channels are cut into blocks of 256, one warp per block, so that lane l of a
// warp owns channels 8l..8l+7 of its block in every stream: all loads are
// 16-byte vectors and the token's x, key and value are each read once.
//
// Reduction order (fixed, and shared with any other kernel that forms these
// sums): for each (stream, block), every lane accumulates its 8 channels in
// order with fmaf starting from 0, the warp combines the 32 lane sums with an
// xor butterfly (16, 8, 4, 2, 1), and the block sums are added in block order
// starting from 0.  Each warp stores its block sums into the shared memory of
// every CTA of the cluster (DSMEM); after one cluster barrier every CTA adds
// them up locally.  The result does not depend on timing, and the
// split-K path rounds kv to bf16 exactly as the separate reduction kernel does,
// so engram_forward and lookup_project + gate_apply agree bit for bit.
#include <cstdlib>

#include "common.cuh"
#include "internal.cuh"

namespace engram {
namespace {

constexpr int kMaxHc = 4;
constexpr int kBlockCh = 256;                    // channels per reduction block (one warp)
constexpr int kMaxBlocks = 5120 / kBlockCh;      // blocks per stream for dim = 5120
constexpr int kGateMaxThreads = kMaxBlocks * 32;
constexpr int kGateSmallThreads = kMaxBlocks / 4 * 32;   // dim = 5120 in clusters of 4

__device__ __forceinline__ void unpack8(uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// A thread's kv values, 8 per group: group s < HC is stream s's key (offset
// s * dim), group kMaxHc the value (offset HC * dim), from the fp32 partial
// sums: summed over the splits in order, then rounded to bf16 (the
// projection's output type).  The loop runs over splits outside and groups
// inside, so each split's loads of all groups are in flight together.
__device__ __forceinline__ bool kv_group(int g, int HC) { return g < HC || g == kMaxHc; }
__device__ __forceinline__ int kv_offset(int g, int HC, int D) { return (g < kMaxHc ? g : HC) * D; }

__device__ __forceinline__ void load_partials(const float* part, int HC, int D, int splits, int64_t split_stride,
                                              float (&f)[kMaxHc + 1][8]) {
#pragma unroll
  for (int g = 0; g < kMaxHc + 1; ++g) {
    if (kv_group(g, HC)) {
      const float4* q = reinterpret_cast<const float4*>(part + kv_offset(g, HC, D));
      const float4 a = __ldg(q), b = __ldg(q + 1);
      f[g][0] = a.x; f[g][1] = a.y; f[g][2] = a.z; f[g][3] = a.w;
      f[g][4] = b.x; f[g][5] = b.y; f[g][6] = b.z; f[g][7] = b.w;
    }
  }
  for (int s = 1; s < splits; ++s) {
    const float* p = part + s * split_stride;
    float4 c[kMaxHc + 1], d[kMaxHc + 1];
#pragma unroll
    for (int g = 0; g < kMaxHc + 1; ++g) {
      if (kv_group(g, HC)) {
        const float4* q = reinterpret_cast<const float4*>(p + kv_offset(g, HC, D));
        c[g] = __ldg(q);
        d[g] = __ldg(q + 1);
      }
    }
#pragma unroll
    for (int g = 0; g < kMaxHc + 1; ++g) {
      if (kv_group(g, HC)) {
        f[g][0] += c[g].x; f[g][1] += c[g].y; f[g][2] += c[g].z; f[g][3] += c[g].w;
        f[g][4] += d[g].x; f[g][5] += d[g].y; f[g][6] += d[g].z; f[g][7] += d[g].w;
      }
    }
  }
#pragma unroll
  for (int g = 0; g < kMaxHc + 1; ++g)
#pragma unroll
    for (int j = 0; j < 8; ++j) f[g][j] = round_bf16(f[g][j]);
}

// The thread's 8 channels of q_weight*k_weight for every stream.
__device__ __forceinline__ void load_wprod(const float* wprod, int HC, int D, int d0, float (&w)[kMaxHc][8]) {
#pragma unroll
  for (int s = 0; s < kMaxHc; ++s) {
    if (s < HC) {
      const float4 w0 = __ldg(reinterpret_cast<const float4*>(wprod + s * D + d0));
      const float4 w1 = __ldg(reinterpret_cast<const float4*>(wprod + s * D + d0) + 1);
      w[s][0] = w0.x; w[s][1] = w0.y; w[s][2] = w0.z; w[s][3] = w0.w;
      w[s][4] = w1.x; w[s][5] = w1.y; w[s][6] = w1.z; w[s][7] = w1.w;
    }
  }
}

// MAX_THREADS bounds the block: 160 for dim = 5120 in clusters of 4 (the
// registers then hold a thread's x, weights and kv at once), kGateMaxThreads
// for other shapes.
template <bool FROM_PARTIALS, int MAX_THREADS>
__global__ void __launch_bounds__(MAX_THREADS) gate_residual_kernel(const GateArgs a) {
  __shared__ float red[kMaxBlocks][3 * kMaxHc];   // every block's sums, pushed by the owning CTAs
  __shared__ float tot[3 * kMaxHc];
  __shared__ float gate_s[kMaxHc];

  const int G = a.cluster;
  const uint32_t rank = G > 1 ? cluster_ctarank() : 0u;
  const int64_t m = blockIdx.x / G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wpc = blockDim.x >> 5;                 // blocks per CTA
  const int nblocks = wpc * G;                     // blocks per stream
  const int D = a.dim;
  const int HC = a.hc;
  const int64_t N = static_cast<int64_t>(D) * (HC + 1);
  const int d0 = (static_cast<int>(rank) * wpc + warp) * kBlockCh + lane * 8;
  const uint16_t* xm = a.x + m * HC * D;
  uint16_t* om = a.out + m * HC * D;

  // x and the mask are inputs of the call, written before the gather ran, so
  // they may be read before the projection has finished
  if (a.mask != nullptr && a.mask[m] == 0) {
    // a masked token leaves the streams as they were: copied, gate 0
    grid_dependency_wait();
    if (om != xm) {
      for (int s = 0; s < HC; ++s)
        *reinterpret_cast<uint4*>(om + s * D + d0) = __ldg(reinterpret_cast<const uint4*>(xm + s * D + d0));
    }
    if (a.gates != nullptr && rank == 0 && threadIdx.x < HC) a.gates[m * HC + threadIdx.x] = 0.0f;
    grid_launch_dependents();
    return;
  }

  // The product q_weight * k_weight is formed when a context is created, long
  // before this kernel, so it is read before the wait too -- unless the caller
  // forms it in the same call (wprod_after_wait: the allocation-free entry
  // point), where it is read after the wait like every other output of an
  // earlier kernel.
  float h[kMaxHc][8], w[kMaxHc][8];
#pragma unroll
  for (int s = 0; s < kMaxHc; ++s)
    if (s < HC) unpack8(__ldg(reinterpret_cast<const uint4*>(xm + s * D + d0)), h[s]);
  if (!a.wprod_after_wait) load_wprod(a.wprod, HC, D, d0, w);

  grid_dependency_wait();        // kv / the partial sums come from the projection
  grid_launch_dependents();
  if (a.wprod_after_wait) load_wprod(a.wprod, HC, D, d0, w);

  float kv[kMaxHc + 1][8];       // the streams' keys, then the value
  if (FROM_PARTIALS) {
    load_partials(a.part + m * N + d0, HC, D, a.splits, a.M * N, kv);
  } else {
#pragma unroll
    for (int g = 0; g < kMaxHc + 1; ++g)
      if (kv_group(g, HC)) unpack8(__ldg(reinterpret_cast<const uint4*>(a.kv + m * N + kv_offset(g, HC, D) + d0)), kv[g]);
  }
  float sums[3 * kMaxHc];
#pragma unroll
  for (int i = 0; i < 3 * kMaxHc; ++i) sums[i] = 0.0f;
#pragma unroll
  for (int s = 0; s < kMaxHc; ++s) {
    if (s < HC) {
      float sh = 0.0f, sk = 0.0f, sd = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        sh = fmaf(h[s][j], h[s][j], sh);
        sk = fmaf(kv[s][j], kv[s][j], sk);
        sd = fmaf(__fmul_rn(h[s][j], w[s][j]), kv[s][j], sd);
      }
      sums[3 * s + 0] = sh;
      sums[3 * s + 1] = sk;
      sums[3 * s + 2] = sd;
    }
  }
  float v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = kv[kMaxHc][j];

  // one block sum per warp: xor butterfly 16, 8, 4, 2, 1
#pragma unroll
  for (int i = 0; i < 3 * kMaxHc; ++i) {
    float x = sums[i];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
    sums[i] = x;
  }
  // every CTA of the cluster receives every block's sums: lane r of the warp
  // stores them into CTA r (remote stores complete before the cluster barrier)
  const int blk = static_cast<int>(rank) * wpc + warp;
  if (G > 1) {
    if (lane < G) {
#pragma unroll
      for (int i = 0; i < 3 * kMaxHc; ++i) st_dsmem_f32(&red[blk][i], static_cast<uint32_t>(lane), sums[i]);
    }
    cluster_arrive();
    cluster_wait();
  } else {
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < 3 * kMaxHc; ++i) red[blk][i] = sums[i];
    }
    __syncthreads();
  }
  if (threadIdx.x < 3 * HC) {            // one (stream, quantity) per thread, blocks in order
    float acc = 0.0f;
    for (int b = 0; b < nblocks; ++b) acc += red[b][threadIdx.x];
    tot[threadIdx.x] = acc;
  }
  __syncthreads();
  if (threadIdx.x < HC) {
    const int t = threadIdx.x;
    const float g = engram_gate(tot[3 * t], tot[3 * t + 1], tot[3 * t + 2], D, a.eps, a.clamp, a.inv_sqrt_dim);
    gate_s[t] = g;
    if (a.gates != nullptr && rank == 0) a.gates[m * HC + t] = g;
  }
  __syncthreads();

#pragma unroll
  for (int s = 0; s < kMaxHc; ++s) {
    if (s < HC) {
      const float g = gate_s[s];
      uint4 o;
      o.x = pack_bf16x2(fmaf(g, v[0], h[s][0]), fmaf(g, v[1], h[s][1]));
      o.y = pack_bf16x2(fmaf(g, v[2], h[s][2]), fmaf(g, v[3], h[s][3]));
      o.z = pack_bf16x2(fmaf(g, v[4], h[s][4]), fmaf(g, v[5], h[s][5]));
      o.w = pack_bf16x2(fmaf(g, v[6], h[s][6]), fmaf(g, v[7], h[s][7]));
      *reinterpret_cast<uint4*>(om + s * D + d0) = o;
    }
  }
}

// The same layer step for bf16 kv as a persistent streaming kernel: one CTA
// per SM walks the tokens blockIdx.x, blockIdx.x + gridDim.x, ...; thread 0
// fetches each token's x and kv rows (contiguous: 40 KB and 50 KB at dim =
// 5120, hc = 4) with two bulk copies into a two-slot shared-memory ring, so
// the next token streams in while this one is gated, and q_weight*k_weight is
// read once per CTA.  Warp w owns blocks w*BPW .. w*BPW+BPW-1 of every stream
// and lane l channels 8l..8l+7 of each, so every block's sums are formed by
// the same lane and warp arithmetic as in gate_residual_kernel, and the block
// sums are added in the same order: the same bits.
template <int BPW>
__global__ void __launch_bounds__(kMaxBlocks / BPW * 32, 1) gate_residual_stream_kernel(const GateArgs a) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[2];
  __shared__ float red[kMaxBlocks][3 * kMaxHc];
  __shared__ float tot[3 * kMaxHc];
  __shared__ float gate_s[kMaxHc];
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int D = a.dim;
  const int HC = a.hc;
  const int nblocks = D / kBlockCh;
  const int64_t N = static_cast<int64_t>(D) * (HC + 1);
  const uint32_t xbytes = static_cast<uint32_t>(HC * D * 2);
  const uint32_t kvbytes = static_cast<uint32_t>(N * 2);
  const uint32_t slot = (xbytes + kvbytes + 127u) & ~127u;
  int d0[BPW];
#pragma unroll
  for (int j = 0; j < BPW; ++j) d0[j] = (warp * BPW + j) * kBlockCh + lane * 8;

  if (threadIdx.x == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    fence_mbarrier_init();
    abort_flag = 0;
  }
  // q_weight * k_weight, once per CTA: before the wait when a context formed
  // it at create time, after it when the caller formed it in the same call
  // (wprod_after_wait)
  float w[BPW][kMaxHc][8];
  if (!a.wprod_after_wait) {
#pragma unroll
    for (int j = 0; j < BPW; ++j) load_wprod(a.wprod, HC, D, d0[j], w[j]);
  }
  __syncthreads();
  grid_dependency_wait();        // kv comes from the projection
  grid_launch_dependents();
  if (a.wprod_after_wait) {
#pragma unroll
    for (int j = 0; j < BPW; ++j) load_wprod(a.wprod, HC, D, d0[j], w[j]);
  }

  const uint64_t pol = policy_evict_first();
  const int64_t step = gridDim.x;
  uint32_t issued[2] = {0u, 0u};   // thread 0: copies issued per slot
  auto fetch = [&](int64_t m, int b) {
    uint8_t* xs = ring + b * slot;
    mbar_arrive_expect_tx(&full[b], xbytes + kvbytes);
    bulk_load_hint(xs, a.x + m * HC * D, xbytes, &full[b], pol);
    bulk_load_hint(xs + xbytes, a.kv + m * N, kvbytes, &full[b], pol);
    ++issued[b];
  };
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b)
      if (blockIdx.x + b * step < a.M) fetch(blockIdx.x + b * step, b);
  }

  int i = 0;
  for (int64_t m = blockIdx.x; m < a.M; m += step, ++i) {
    const int b = i & 1;
    const bool ok = mbar_wait(&full[b], static_cast<uint32_t>((i >> 1) & 1), &abort_flag);
    if (!ok && threadIdx.x == 0) {
      abort_flag = 1;
      atomicOr(a.err, kErrTimeout);
    }
    __syncthreads();
    if (abort_flag) break;
    const uint32_t xs = smem_u32(ring + b * slot);
    const uint32_t ks = xs + xbytes;
    uint16_t* om = a.out + m * HC * D;

    if (a.mask != nullptr && a.mask[m] == 0) {
      // a masked token leaves the streams as they were: copied, gate 0
#pragma unroll
      for (int j = 0; j < BPW; ++j)
        for (int s = 0; s < HC; ++s)
          *reinterpret_cast<uint4*>(om + s * D + d0[j]) = ld_shared_v4(xs + 2u * static_cast<uint32_t>(s * D + d0[j]));
      if (a.gates != nullptr && threadIdx.x < HC) a.gates[m * HC + threadIdx.x] = 0.0f;
    } else {
#pragma unroll
      for (int j = 0; j < BPW; ++j) {
        float sums[3 * kMaxHc];
#pragma unroll
        for (int s = 0; s < kMaxHc; ++s) {
          sums[3 * s] = sums[3 * s + 1] = sums[3 * s + 2] = 0.0f;
          if (s < HC) {
            float h[8], k[8];
            unpack8(ld_shared_v4(xs + 2u * static_cast<uint32_t>(s * D + d0[j])), h);
            unpack8(ld_shared_v4(ks + 2u * static_cast<uint32_t>(s * D + d0[j])), k);
            float sh = 0.0f, sk = 0.0f, sd = 0.0f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              sh = fmaf(h[c], h[c], sh);
              sk = fmaf(k[c], k[c], sk);
              sd = fmaf(__fmul_rn(h[c], w[j][s][c]), k[c], sd);
            }
            sums[3 * s] = sh;
            sums[3 * s + 1] = sk;
            sums[3 * s + 2] = sd;
          }
        }
#pragma unroll
        for (int q = 0; q < 3 * kMaxHc; ++q) {
          float v = sums[q];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
          if (lane == 0) red[warp * BPW + j][q] = v;
        }
      }
      __syncthreads();
      if (threadIdx.x < 3 * HC) {        // one (stream, quantity) per thread, blocks in order
        float acc = 0.0f;
        for (int blk = 0; blk < nblocks; ++blk) acc += red[blk][threadIdx.x];
        tot[threadIdx.x] = acc;
      }
      __syncthreads();
      if (threadIdx.x < HC) {
        const int t = threadIdx.x;
        const float g = engram_gate(tot[3 * t], tot[3 * t + 1], tot[3 * t + 2], D, a.eps, a.clamp, a.inv_sqrt_dim);
        gate_s[t] = g;
        if (a.gates != nullptr) a.gates[m * HC + t] = g;
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < BPW; ++j) {
        float v[8];
        unpack8(ld_shared_v4(ks + 2u * static_cast<uint32_t>(HC * D + d0[j])), v);
#pragma unroll
        for (int s = 0; s < kMaxHc; ++s) {
          if (s < HC) {
            const float g = gate_s[s];
            float h[8];
            unpack8(ld_shared_v4(xs + 2u * static_cast<uint32_t>(s * D + d0[j])), h);
            uint4 o;
            o.x = pack_bf16x2(fmaf(g, v[0], h[0]), fmaf(g, v[1], h[1]));
            o.y = pack_bf16x2(fmaf(g, v[2], h[2]), fmaf(g, v[3], h[3]));
            o.z = pack_bf16x2(fmaf(g, v[4], h[4]), fmaf(g, v[5], h[5]));
            o.w = pack_bf16x2(fmaf(g, v[6], h[6]), fmaf(g, v[7], h[7]));
            *reinterpret_cast<uint4*>(om + s * D + d0[j]) = o;
          }
        }
      }
    }
    __syncthreads();                     // slot b and gate_s are free again
    if (threadIdx.x == 0 && m + 2 * step < a.M) fetch(m + 2 * step, b);
  }
  if (threadIdx.x == 0 && abort_flag) {
    // let every copy already issued land before the CTA can exit
    for (int b = 0; b < 2; ++b)
      if (issued[b] > 0) mbar_wait(&full[b], (issued[b] - 1u) & 1u, nullptr, kDrainLimitNs);
  }
}

__global__ void reduce_partials_kernel(const float* __restrict__ part, int splits, int64_t MN,
                                       uint16_t* __restrict__ kv) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t n4 = MN >> 2;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 a = __ldg(reinterpret_cast<const float4*>(part) + i);
    for (int s = 1; s < splits; ++s) {
      const float4 c = __ldg(reinterpret_cast<const float4*>(part + s * MN) + i);
      a.x += c.x; a.y += c.y; a.z += c.z; a.w += c.w;
    }
    uint2 o;
    o.x = pack_bf16x2(a.x, a.y);
    o.y = pack_bf16x2(a.z, a.w);
    reinterpret_cast<uint2*>(kv)[i] = o;
  }
}

__global__ void weight_product_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                                      float* __restrict__ w, int64_t n) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    w[i] = __fmul_rn(bf16_bits_to_float(q[i]), bf16_bits_to_float(k[i]));
}

}  // namespace

int gate_cluster_size(int dim) {
  const int nblocks = dim / kBlockCh;
  return nblocks % 4 == 0 ? 4 : (nblocks % 2 == 0 ? 2 : 1);
}

// Shared memory of the streaming kernel: two slots of one token's x and kv.
size_t gate_stream_smem(int dim, int hc) {
  const size_t slot = (static_cast<size_t>(hc) * dim * 2 + static_cast<size_t>(hc + 1) * dim * 2 + 127) & ~size_t{127};
  return 2 * slot;
}

// Batches of at least this many tokens (with bf16 kv) take the streaming
// kernel, smaller ones spread each token over a cluster for latency.  Measured
// on GB300 inside a layer step against the one-CTA-per-token kernel it
// replaced: 512 tokens 137.6 -> 136.0 us, 4,096 tokens 862 -> 844 us, 16,384
// tokens 3.35 -> 3.27 ms (that kernel in turn had taken 512 tokens from 25.3 to
// 20.5 us, 4,096 tokens from 167 to 98 us against the cluster kernel).
// ENGRAM_GATE_STREAM_MIN overrides the threshold for measurements.
int64_t gate_stream_min_tokens() {
  static const int64_t v = [] {
    const char* e = std::getenv("ENGRAM_GATE_STREAM_MIN");
    return e != nullptr ? static_cast<int64_t>(std::atoll(e)) : int64_t{256};
  }();
  return v;
}

cudaError_t gate_prepare() {
  const int smem = static_cast<int>(gate_stream_smem(5120, kMaxHc));
  cudaError_t e = cudaFuncSetAttribute(gate_residual_stream_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gate_residual_stream_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  return e;
}

cudaError_t launch_gate(const GateArgs& a_in, cudaStream_t stream) {
  if (a_in.M == 0) return cudaSuccess;
  GateArgs a = a_in;
  const int nblocks = a.dim / kBlockCh;
  if (a.part == nullptr && a.err != nullptr && a.num_sms > 0 && a.M >= gate_stream_min_tokens()) {
    a.cluster = 1;
    const size_t smem = gate_stream_smem(a.dim, a.hc);
    const dim3 grid(static_cast<unsigned>(a.M < a.num_sms ? a.M : a.num_sms));
    if (nblocks % 2 == 0)
      return launch_pdl(gate_residual_stream_kernel<2>, grid, dim3(static_cast<unsigned>(nblocks / 2 * 32)), smem,
                        stream, 1, a);
    return launch_pdl(gate_residual_stream_kernel<1>, grid, dim3(static_cast<unsigned>(nblocks * 32)), smem, stream,
                      1, a);
  }
  a.cluster = gate_cluster_size(a.dim);
  const unsigned threads = static_cast<unsigned>(a.dim / kBlockCh / a.cluster * 32);
  const dim3 grid(static_cast<unsigned>(a.M * a.cluster));
  if (threads <= kGateSmallThreads) {
    if (a.part != nullptr)
      return launch_pdl(gate_residual_kernel<true, kGateSmallThreads>, grid, dim3(threads), 0, stream, a.cluster, a);
    return launch_pdl(gate_residual_kernel<false, kGateSmallThreads>, grid, dim3(threads), 0, stream, a.cluster, a);
  }
  if (a.part != nullptr)
    return launch_pdl(gate_residual_kernel<true, kGateMaxThreads>, grid, dim3(threads), 0, stream, a.cluster, a);
  return launch_pdl(gate_residual_kernel<false, kGateMaxThreads>, grid, dim3(threads), 0, stream, a.cluster, a);
}

cudaError_t launch_reduce_partials(const float* part, int32_t splits, int64_t M, int32_t N, uint16_t* kv,
                                   int num_sms, cudaStream_t stream) {
  const int64_t MN = M * N;
  if (MN == 0) return cudaSuccess;
  int64_t blocks = (MN / 4 + 255) / 256;
  if (blocks > static_cast<int64_t>(num_sms) * 8) blocks = static_cast<int64_t>(num_sms) * 8;
  return launch_pdl(reduce_partials_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, 1, part,
                    splits, MN, kv);
}

cudaError_t launch_weight_product(const uint16_t* q, const uint16_t* k, float* wprod, int64_t n,
                                  cudaStream_t stream) {
  weight_product_kernel<<<64, 256, 0, stream>>>(q, k, wprod, n);
  return cudaGetLastError();
}

}  // namespace engram
