// The n-gram hash that turns token ids into the table rows of every Engram
// layer (atlas.klimoza.dev "deepseek-v4.1 / engram-second", the hash `forward`
// excerpt; monishver11.github.io "DeepSeek's Other Modules", section "The
// lookup pipeline").  Look-back ids inside this call's chunk are recomputed
// from the input ids and ids before it are read from the session cache, so no
// thread reads a cache entry another thread of the same call writes.
// Integer-only; the products wrap at 64 bits like int64 tensors.
#include "../../include/engram.h"
#include "common.cuh"
#include "internal.cuh"

using namespace engram;

namespace {

constexpr int kMaxNgram = 8;
constexpr int kMaxPrimes = 6144;   // Barrett multipliers held in 48 KB of shared memory

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

// Remainder of a signed 64-bit hash by a positive prime p, with the divisor's
// sign (Python / torch `%`): Barrett reduction (Barrett, "Implementing the
// Rivest Shamir and Adleman public key encryption algorithm on a standard
// digital signal processor", CRYPTO '86) of |x| with m = floor((2^64-1)/p).
// q = floor(|x| m / 2^64) lies in (|x|/p - 2, |x|/p], so |x| - q p < 2p and one
// conditional subtraction finishes it.
__device__ __forceinline__ int64_t floor_mod(int64_t x, uint64_t p, uint64_t m) {
  const uint64_t ax = x < 0 ? 0ull - static_cast<uint64_t>(x) : static_cast<uint64_t>(x);
  uint64_t r = ax - __umul64hi(ax, m) * p;
  if (r >= p) r -= p;
  if (x < 0 && r != 0) r = p - r;
  return static_cast<int64_t>(r);
}

// One thread per output element, indexed like the output array
// [n_layers, B, L, cols] so that stores are coalesced: it forms its token's
// look-back ids (the threads of a token share them through L1), the rolling
// hash up to its column's n-gram order, and one remainder.  The block first
// turns every prime into its Barrett multiplier in shared memory.  Idx is the
// index type: 32-bit when the output has fewer than 2^31 elements.
template <typename Idx>
__global__ void __launch_bounds__(256) ngram_hash_kernel(const HashArgs a) {
  extern __shared__ uint64_t barrett[];
  const int n_primes = a.n_layers * (a.n - 1) * a.heads;
  grid_dependency_wait();
  grid_launch_dependents();
  for (int j = threadIdx.x; j < n_primes; j += blockDim.x) barrett[j] = ~0ull / static_cast<uint64_t>(__ldg(a.primes + j));
  __syncthreads();
  const Idx cols = static_cast<Idx>((a.n - 1) * a.heads);
  const Idx tokens = static_cast<Idx>(a.B * a.L);
  const Idx L = static_cast<Idx>(a.L);
  const Idx total = tokens * static_cast<Idx>(a.n_layers) * cols;
  for (Idx i = static_cast<Idx>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<Idx>(gridDim.x) * blockDim.x) {
    const Idx row = i / cols;
    const int c = static_cast<int>(i - row * cols);
    const int g = static_cast<int>(row / tokens);
    const Idx t = row - static_cast<Idx>(g) * tokens;
    const int64_t b = static_cast<int64_t>(t / L);
    const int64_t l = static_cast<int64_t>(t) - b * a.L;
    const int64_t pos = a.start_pos + l;
    const int k = c / a.heads + 1;                   // this column hashes the (k+1)-gram
    const int64_t* mul = a.multipliers + g * a.n;
    uint64_t rolling = 0;
    bool blocked = false;
    for (int s = 0; s <= k; ++s) {
      const int64_t p = pos - s;
      int32_t src = a.dead_id;
      if (p >= a.start_pos) {
        src = compress(a, b, p - a.start_pos);
      } else if (p >= 0) {
        src = a.cache[b * a.max_len + p];
      }
      blocked = blocked || p < 0 || src == a.dead_id;
      const int64_t tok = blocked ? a.pad_id : src;
      rolling ^= static_cast<uint64_t>(tok) * static_cast<uint64_t>(__ldg(mul + s));
    }
    const int j = g * static_cast<int>(cols) + c;    // primes and offsets share the column order
    a.out[i] = floor_mod(static_cast<int64_t>(rolling), static_cast<uint64_t>(__ldg(a.primes + j)), barrett[j]) +
               __ldg(a.offsets + j);
    if (g == 0 && c == 0) a.cache[b * a.max_len + pos] = compress(a, b, l);
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
  if (int64_t{c.n_layers} * (c.max_ngram_size - 1) * c.n_heads > kMaxPrimes) return ENGRAM_EUNSUPPORTED;
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
  const int64_t total = B * L * c.n_layers * (c.max_ngram_size - 1) * c.n_heads;
  const size_t smem = static_cast<size_t>(c.n_layers) * (c.max_ngram_size - 1) * c.n_heads * sizeof(uint64_t);
  int64_t blocks = (total + 255) / 256;
  if (blocks > static_cast<int64_t>(sms) * 8) blocks = static_cast<int64_t>(sms) * 8;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e =
      total < (int64_t{1} << 31)
          ? launch_pdl(ngram_hash_kernel<uint32_t>, dim3(static_cast<unsigned>(blocks)), dim3(256), smem, st, 1, a)
          : launch_pdl(ngram_hash_kernel<uint64_t>, dim3(static_cast<unsigned>(blocks)), dim3(256), smem, st, 1, a);
  return e == cudaSuccess ? ENGRAM_OK : ENGRAM_ECUDA;
}
