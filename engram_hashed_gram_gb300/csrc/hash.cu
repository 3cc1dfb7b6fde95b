// The n-gram hash that turns token ids into the table rows of every Engram
// layer (atlas.klimoza.dev "deepseek-v4.1 / engram-second", the hash `forward`
// excerpt; monishver11.github.io "DeepSeek's Other Modules", section "The
// lookup pipeline").  One thread per (sequence, position): it compresses its
// token, stores it in the session cache, forms the blocked look-back ids (ids
// inside this call's chunk are recomputed from the input ids, ids before it are
// read from the cache, so no thread reads a cache entry another thread of the
// same call writes), and writes the n_layers x (max_ngram_size-1) x n_heads
// rows.  Integer-only; the products wrap at 64 bits like int64 tensors.
#include "../../include/engram.h"
#include "common.cuh"
#include "internal.cuh"

using namespace engram;

namespace {

constexpr int kMaxNgram = 8;

struct HashArgs {
  const int32_t* token_map;
  const int64_t* multipliers;
  const int64_t* primes;
  const int64_t* offsets;
  int32_t* cache;
  const int64_t* ids;
  const uint8_t* mask;
  int64_t* out;
  int64_t start_pos;
  int64_t B;
  int64_t L;
  int64_t max_len;
  int64_t vocab;
  int32_t n_layers;
  int32_t n;
  int32_t heads;
  int32_t pad_id;
  int32_t dead_id;
};

__device__ __forceinline__ int32_t compress(const HashArgs& a, int64_t b, int64_t l) {
  const int64_t t = a.ids[b * a.L + l];
  int32_t c = (t >= 0 && t < a.vocab) ? __ldg(a.token_map + t) : a.dead_id;
  if (a.mask != nullptr && a.mask[b * a.L + l] == 0) c = a.dead_id;
  return c;
}

__global__ void __launch_bounds__(256) ngram_hash_kernel(const HashArgs a) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t total = a.B * a.L;
  const int cols = (a.n - 1) * a.heads;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t b = i / a.L;
    const int64_t l = i - b * a.L;
    const int64_t pos = a.start_pos + l;
    int64_t tok[kMaxNgram];
    bool blocked = false;
    for (int s = 0; s < a.n; ++s) {
      const int64_t p = pos - s;
      int32_t src = a.dead_id;
      if (p >= a.start_pos) {
        src = compress(a, b, p - a.start_pos);
      } else if (p >= 0) {
        src = a.cache[b * a.max_len + p];
      }
      blocked = blocked || p < 0 || src == a.dead_id;
      tok[s] = blocked ? a.pad_id : src;
    }
    a.cache[b * a.max_len + pos] = compress(a, b, l);
    for (int g = 0; g < a.n_layers; ++g) {
      const int64_t* mul = a.multipliers + g * a.n;
      uint64_t rolling = static_cast<uint64_t>(tok[0]) * static_cast<uint64_t>(__ldg(mul));
      int64_t* o = a.out + ((static_cast<int64_t>(g) * a.B + b) * a.L + l) * cols;
      for (int k = 1; k < a.n; ++k) {
        rolling ^= static_cast<uint64_t>(tok[k]) * static_cast<uint64_t>(__ldg(mul + k));
        const int64_t h = static_cast<int64_t>(rolling);
        for (int j = 0; j < a.heads; ++j) {
          const int c = (k - 1) * a.heads + j;
          const int64_t prime = __ldg(a.primes + (static_cast<int64_t>(g) * (a.n - 1) + (k - 1)) * a.heads + j);
          int64_t r = h % prime;
          if (r < 0) r += prime;
          o[c] = r + __ldg(a.offsets + static_cast<int64_t>(g) * cols + c);
        }
      }
    }
  }
}

bool aligned(const void* p, uintptr_t al) { return (reinterpret_cast<uintptr_t>(p) & (al - 1)) == 0; }

}  // namespace

extern "C" engram_status engram_hash(const engram_hash_config* cfg, const int32_t* token_map,
                                     const int64_t* multipliers, const int64_t* primes, const int64_t* offsets,
                                     int32_t* cache, const int64_t* input_ids, const uint8_t* token_mask,
                                     int64_t start_pos, int64_t* hash_ids, int64_t B, int64_t L,
                                     engram_stream_t stream) {
  if (cfg == nullptr) return ENGRAM_EINVAL;
  const engram_hash_config& c = *cfg;
  if (c.n_layers <= 0 || c.max_ngram_size < 2 || c.max_ngram_size > kMaxNgram || c.n_heads <= 0 || c.n_heads > 32 ||
      c.max_batch < 0 || c.max_len < 0 || c.vocab_size < 0)
    return ENGRAM_EINVAL;
  if (B < 0 || L < 0 || start_pos < 0 || B > c.max_batch || L > c.max_len || start_pos > c.max_len - L)
    return ENGRAM_EINVAL;
  if (B == 0 || L == 0) return ENGRAM_OK;
  if (token_map == nullptr || multipliers == nullptr || primes == nullptr || offsets == nullptr || cache == nullptr ||
      input_ids == nullptr || hash_ids == nullptr)
    return ENGRAM_EINVAL;
  if (!aligned(token_map, 4) || !aligned(cache, 4) || !aligned(multipliers, 8) || !aligned(primes, 8) ||
      !aligned(offsets, 8) || !aligned(input_ids, 8) || !aligned(hash_ids, 8))
    return ENGRAM_EINVAL;
  HashArgs a{};
  a.token_map = token_map;
  a.multipliers = multipliers;
  a.primes = primes;
  a.offsets = offsets;
  a.cache = cache;
  a.ids = input_ids;
  a.mask = token_mask;
  a.out = hash_ids;
  a.start_pos = start_pos;
  a.B = B;
  a.L = L;
  a.max_len = c.max_len;
  a.vocab = c.vocab_size;
  a.n_layers = c.n_layers;
  a.n = c.max_ngram_size;
  a.heads = c.n_heads;
  a.pad_id = c.pad_id;
  a.dead_id = c.dead_id;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return ENGRAM_ECUDA;
  int64_t blocks = (B * L + 255) / 256;
  if (blocks > static_cast<int64_t>(sms) * 8) blocks = static_cast<int64_t>(sms) * 8;
  const cudaError_t e = launch_pdl(ngram_hash_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                                   reinterpret_cast<cudaStream_t>(stream), 1, a);
  return e == cudaSuccess ? ENGRAM_OK : ENGRAM_ECUDA;
}
