// engram_forward_noalloc: the whole layer for small batches (at most
// ENGRAM_NOALLOC_MAX_TOKENS tokens) with no context and no allocation.
//
// Some callers cannot allocate device memory: a serving engine that reserves
// nearly all of HBM up front for weights and its KV cache and routes every
// other byte through its own allocator, or a plugin whose host process owns the
// GPU's memory budget, cannot let a library call cudaMalloc (and could not
// accept the failure or the implicit synchronisation it may bring).  For them
// this entry point keeps its scratch -- the gathered rows, the split-K partial
// sums (or the bf16 kv), q_weight*k_weight and the device error word -- in one
// file-scope static __device__ array, which the CUDA driver places in device
// memory when it loads this module on a device; every device that loads it
// keeps those bytes until the process exits.
//
// The kernels are the same as engram_forward's (gather/dequant, tcgen05
// projection, gate + residual); only where their scratch lives differs.
#include <cmath>
#include <mutex>

#include "../../include/engram.h"
#include "common.cuh"
#include "internal.cuh"

using namespace engram;

namespace {

constexpr int64_t kMaxTokens = ENGRAM_NOALLOC_MAX_TOKENS;
constexpr int64_t kMaxK = 6144;           // n_cols * head_dim
constexpr int64_t kMaxN = 25600;          // dim * (hc_mult + 1)
constexpr int64_t kMaxHcDim = 4 * 5120;   // hc_mult * dim
constexpr int32_t kMaxSplits = 3;            // sizes the partial sums at the V4.1 shape

constexpr size_t align256(size_t b) { return (b + 255) & ~size_t(255); }
constexpr size_t kErrBytes = 256;
constexpr size_t kWprodBytes = align256(kMaxHcDim * sizeof(float));
constexpr size_t kRowsBytes = align256(kMaxTokens * kMaxK * 2);
constexpr size_t kPartBytes = align256(size_t(kMaxSplits) * kMaxTokens * kMaxN * sizeof(float));
constexpr size_t kScratchBytes = kErrBytes + kWprodBytes + kRowsBytes + kPartBytes;
static_assert(kScratchBytes == ENGRAM_NOALLOC_SCRATCH_BYTES, "header and implementation disagree");

// The scratch.  In host code this name is only a stand-in and must not be
// handed to a kernel; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

// The driver's id of the context current on this thread (0 if none, or if the
// driver entry points are unavailable).  Ids are never reused within a
// process, unlike context handles.
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

struct ScratchSlot {
  unsigned long long context_id;   // the context the address belongs to
  unsigned char* address;
};
std::mutex g_mu;
ScratchSlot g_slots[kMaxDevices] = {};

// Device address of g_scratch on device `dev` (which must be current).  The
// address is looked up (cudaGetSymbolAddress, which also loads this module on
// the device) at the first call on a device and again whenever the device's
// context has changed since (after cudaDeviceReset the module, and with it the
// array, lives at a new address); otherwise the cached address is used.
cudaError_t scratch_address(int dev, unsigned char** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchSlot& slot = g_slots[dev];
  const unsigned long long id = current_context_id();
  if (slot.address == nullptr || id == 0 || slot.context_id != id) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    slot.address = static_cast<unsigned char*>(p);
    slot.context_id = current_context_id();   // the lookup made the device's context current
  }
  *out = slot.address;
  return cudaSuccess;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" engram_status engram_forward_noalloc(const engram_config* cfg, const engram_weights* w,
                                                const int64_t* hash_ids, const uint16_t* x,
                                                const uint8_t* token_mask, uint16_t* out, int64_t B, int64_t T,
                                                engram_stream_t stream) {
  if (cfg == nullptr || w == nullptr) return ENGRAM_EINVAL;
  const engram_config& c = *cfg;
  if (B < 0 || T < 0 || (B != 0 && T > INT64_MAX / B)) return ENGRAM_EINVAL;
  const int64_t M = B * T;
  if (M > kMaxTokens) return ENGRAM_EINVAL;   // the static scratch holds ENGRAM_NOALLOC_MAX_TOKENS tokens
  if (c.dim <= 0 || c.hc_mult <= 0 || c.n_cols <= 0 || c.head_dim <= 0 || c.scale_block <= 0 || c.num_rows < 0 ||
      !(c.eps >= 0.0f) || !(c.clamp >= 0.0f) || c.row_offset < 0 || c.row_offset > INT64_MAX - c.num_rows)
    return ENGRAM_EINVAL;
  if (c.scale_fmt != ENGRAM_SCALE_F32 && c.scale_fmt != ENGRAM_SCALE_E8M0) return ENGRAM_EUNSUPPORTED;
  if (c.wkv_fmt != ENGRAM_WKV_BF16) return ENGRAM_EUNSUPPORTED;   // the MXFP8 weight needs a context's packed copy
  if (c.dim % kBN != 0 || c.dim > 5120 || c.hc_mult > 4 || c.head_dim % 16 != 0 || c.head_dim % c.scale_block != 0 ||
      c.scale_block % 16 != 0)
    return ENGRAM_EUNSUPPORTED;
  const int64_t K = static_cast<int64_t>(c.n_cols) * c.head_dim;
  const int64_t N = static_cast<int64_t>(c.dim) * (c.hc_mult + 1);
  if (K % kBK != 0 || K > kMaxK || N > kMaxN) return ENGRAM_EUNSUPPORTED;
  if (M == 0) return ENGRAM_OK;
  if (w->table == nullptr || w->scale == nullptr || w->wkv == nullptr || w->q_weight == nullptr ||
      w->k_weight == nullptr || hash_ids == nullptr || x == nullptr || out == nullptr)
    return ENGRAM_EINVAL;
  if (!aligned(w->table, 16) || !aligned(w->wkv, 16) || !aligned(w->q_weight, 2) || !aligned(w->k_weight, 2) ||
      !aligned(w->scale, c.scale_fmt == ENGRAM_SCALE_F32 ? 4 : 1) || !aligned(hash_ids, 8) || !aligned(x, 16) ||
      !aligned(out, 16))
    return ENGRAM_EINVAL;

  int dev = 0, sms = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return ENGRAM_ECUDA;
  if (major != 10 || minor != 3) return ENGRAM_EUNSUPPORTED;
  // Every buffer the kernels will dereference must be readable by this device
  // where it is: a pageable host pointer or another device's memory would make
  // the first kernel that touches it fault.  Nothing is queued before this.
  if (!device_readable(w->table, dev) || !device_readable(w->scale, dev) || !device_readable(w->wkv, dev) ||
      !device_readable(w->q_weight, dev) || !device_readable(w->k_weight, dev))
    return ENGRAM_EINVAL;
  unsigned char* base = nullptr;
  if (scratch_address(dev, &base) != cudaSuccess) return ENGRAM_ECUDA;
  auto* err = reinterpret_cast<unsigned long long*>(base);
  auto* wprod = reinterpret_cast<float*>(base + kErrBytes);
  auto* rows = reinterpret_cast<uint16_t*>(base + kErrBytes + kWprodBytes);
  auto* part = reinterpret_cast<float*>(base + kErrBytes + kWprodBytes + kRowsBytes);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  // the split-K factor: engram_forward's rule (whole-K tiles once they fill
  // 5/8 of the grid in one wave, since they stream the weight at the HBM rate;
  // otherwise the factor in {2, 3, 4, 6, 8} that minimises waves x K blocks),
  // among the factors whose fp32 partial sums fit the scratch
  const int32_t m_tiles = static_cast<int32_t>((M + kBM - 1) / kBM);
  const int32_t n_tiles = static_cast<int32_t>(N / kBN);
  const int32_t kbt = static_cast<int32_t>(K / kBK);
  const int64_t tiles = static_cast<int64_t>(m_tiles) * n_tiles;
  auto waves = [&](int64_t u) { return (u + sms - 1) / sms; };
  int32_t splits = 1;
  int64_t best = waves(tiles) * kbt;
  const bool streams_whole = tiles <= sms && tiles * 8 >= static_cast<int64_t>(sms) * 5;
  const int32_t cand[] = {2, 3, 4, 6, 8};
  for (int32_t sp : cand) {
    if (streams_whole || kbt % sp != 0) continue;
    if (static_cast<size_t>(sp) * M * N * sizeof(float) > kPartBytes) continue;
    const int64_t cost = waves(tiles * sp) * (kbt / sp);
    if (cost < best) {
      best = cost;
      splits = sp;
    }
  }

  // the error word is the only scratch that must start at zero; the rest is
  // overwritten before it is read
  if (cudaMemsetAsync(err, 0, 2 * sizeof(unsigned long long), s) != cudaSuccess) return ENGRAM_ECUDA;
  // q_weight*k_weight is formed on every call, into the scratch.  Ordering: the
  // gather waits (griddepcontrol.wait) for this kernel; the projection waits
  // for the gather; the gate kernel reads the product only after its own wait
  // (wprod_after_wait below), so no kernel of this call reads it early, and the
  // previous call's product left in the array is never read.
  if (launch_weight_product(w->q_weight, w->k_weight, wprod, static_cast<int64_t>(c.hc_mult) * c.dim, s) !=
      cudaSuccess)
    return ENGRAM_ECUDA;

  GatherArgs g{};
  g.ids = hash_ids;
  g.table = w->table;
  g.scale = w->scale;
  g.out = rows;
  g.rows_total = M * c.n_cols;
  g.R = c.num_rows;
  g.row0 = c.row_offset;
  g.head_dim = c.head_dim;
  g.scale_block = c.scale_block;
  g.scale_fmt = c.scale_fmt;
  g.check_ids = 0;
  g.err = err;
  if (launch_gather(g, sms, s) != cudaSuccess) return ENGRAM_ECUDA;

  CUtensorMap tmB;
  if (!make_tmap_bf16(&tmB, w->wkv, static_cast<uint64_t>(N), static_cast<uint64_t>(K), kBN)) return ENGRAM_ECUDA;
  GemmArgs a{};
  a.M = M;
  a.N = static_cast<int32_t>(N);
  a.K = static_cast<int32_t>(K);
  a.splits = splits;
  a.kb_per_split = kbt / splits;
  a.m_tiles = m_tiles;
  a.n_tiles = n_tiles;
  a.group_m = m_tiles;
  a.units = tiles * splits;
  a.out_mode = splits == 1 ? kOutBf16 : kOutPartial;
  a.kv = reinterpret_cast<uint16_t*>(part);   // splits == 1: bf16 kv in the partials' space
  a.part = part;
  a.err = err;
  if (gemm_prepare() != cudaSuccess) return ENGRAM_ECUDA;
  const int ctas = static_cast<int>(a.units < sms ? a.units : sms);
  if (launch_gemm(rows, tmB, a, ctas, s) != cudaSuccess) return ENGRAM_ECUDA;

  GateArgs ga{};
  ga.x = x;
  ga.mask = token_mask;
  ga.wprod = wprod;
  ga.out = out;
  ga.gates = nullptr;
  ga.M = M;
  ga.dim = c.dim;
  ga.hc = c.hc_mult;
  ga.eps = c.eps;
  ga.clamp = c.clamp;
  ga.inv_sqrt_dim = static_cast<float>(1.0 / std::sqrt(static_cast<double>(c.dim)));
  ga.wprod_after_wait = 1;                    // formed by this call's first kernel
  if (splits == 1) {
    ga.kv = reinterpret_cast<const uint16_t*>(part);
  } else {
    ga.part = part;
    ga.splits = splits;
  }
  return launch_gate(ga, s) == cudaSuccess ? ENGRAM_OK : ENGRAM_ECUDA;
}
