// C ABI of the Engram layer (include/engram.h): argument checks, scratch
// ownership, the projection's work plan and the launch sequence
//   gather/dequant (or, for the MXFP8 weight, gather of codes and scales)
//   -> tcgen05 projection [-> reduction of remainder-split tiles]
//   -> gate + residual (from kv, or from the split-K partial sums)
// on the caller's stream, chained by programmatic dependent launch.  No step
// runs on the host.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "../../include/engram.h"
#include "common.cuh"
#include "internal.cuh"

using namespace engram;

struct engram_ctx {
  engram_config cfg;
  engram_weights w;
  int device;
  int num_sms;
  int pair_slots;             // CTA pairs of the pair projection that fit at once (0: not used)
  int sm_budget;              // SMs the projection's persistent grid may occupy (engram_set_sm_budget)
  int32_t test_hooks;         // engram_test_hook bits
  int32_t K;
  int32_t N;
  float* wprod;               // [hc, dim] fp32
  uint16_t* rows;             // [max_tokens, K] bf16 gathered rows
  uint16_t* kv;               // [max_tokens, N] bf16
  float* part;                // [kMaxSplits, part_tokens, N] fp32
  int64_t part_tokens;
  unsigned long long* err;    // device [2]
  float* gsum;                // [max_tokens, hc, dim/256, 4] fused-epilogue block sums
  float* gates;               // [max_tokens, 4] fused-epilogue gates
  uint32_t* counters;         // [ceil(max_tokens/128), 8] fused-epilogue counters and flags
  uint32_t* tickets;          // [2] fused-epilogue work tickets (0 between launches)
  float* rem_ws;              // [num_sms * 4, 128, 256] remainder-split partial tiles (batches > 128 only)
  uint8_t* wpack;             // wkv in 32 KB swizzled tiles (launch_pack_wkv): N*K*2 bytes, N*K for MXFP8
  bool fp8;                   // MXFP8 weight: block-scaled FP8 projection
  uint8_t* wsf;               // fp8: the weight's scales, packed (launch_pack_sfb), N*K/32 bytes
  uint8_t* codes;             // fp8: [max_tokens, K] gathered e4m3 codes
  uint8_t* sfa;               // fp8: [ceil(max_tokens/128), K/128, 512] gathered scales
  CUtensorMap tmW;
  cudaEvent_t* ev;            // stage timing: 4 events per remembered call (null unless enabled)
  int32_t timing_sets;        // calls remembered
  int64_t timing_calls;       // calls timed since enabled
  bool timing;
};

namespace {

constexpr int kMaxSplits = 8;
constexpr int64_t kSplitMaxTokens = 128;   // split-K only while one M tile covers the batch

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct Plan {
  int32_t splits;
  int32_t ctas;
  int32_t m_tiles;
  int32_t n_tiles;
  int64_t units;
  int32_t rem_tiles;    // tiles of the partial last wave cut into K ranges (0: none)
  int32_t rem_splits;
  bool pair;            // CTA pairs (tcgen05 cta_group::2): units are 256 x 256 tiles
};

constexpr int kMaxRemSplits = 4;

// engram_config.fuse_gate: 0 = the library decides by batch size, 1 = the
// fused gate epilogue whenever the plan allows it, -1 = never.
constexpr int32_t kMaxTimedCalls = 4096;     // calls engram_enable_stage_timing can remember
constexpr int32_t kFuseAuto = 0;
constexpr int32_t kFuseAlways = 1;

// Batches of at least this many tokens take the fused gate epilogue when
// fuse_gate is 0 (ENGRAM_FUSE_MIN overrides it for measurements).
// The library's choice (fuse_gate 0) fuses the gate into the CTA-pair
// projection's epilogue from this many tokens on (ENGRAM_FUSE_MIN overrides it
// for measurements).  Measured on GB300, one forward, fused against the
// separate gate kernel: 512 tokens 148 / 131 us, 768 184 / 174, 1,024 236 /
// 241, 2,048 392 / 418, 4,096 742 / 796, 8,192 1,455 / 1,579.  Below that the
// value tiles' wait for all key tiles of their rows is not hidden.
int64_t fuse_auto_min_tokens() {
  static const int64_t v = [] {
    const char* e = std::getenv("ENGRAM_FUSE_MIN");
    return e != nullptr ? static_cast<int64_t>(std::atoll(e)) : int64_t{1024};
  }();
  return v;
}

// Batches of at least this many tokens (bf16 weight) are projected by CTA
// pairs (ENGRAM_PAIR_MIN overrides it for measurements; 0 turns the pairs off).
int64_t pair_min_tokens() {
  static const int64_t v = [] {
    const char* e = std::getenv("ENGRAM_PAIR_MIN");
    const int64_t x = e != nullptr ? static_cast<int64_t>(std::atoll(e)) : int64_t{256};
    return x <= 0 ? INT64_MAX : x;
  }();
  return v;
}

// Whether a batch of M tokens may take the CTA-pair projection: bf16 weight,
// all SMs (no run-ahead budget), and pairs that fit on the device.
bool pair_eligible(const engram_ctx* c, int64_t M) {
  return !c->fp8 && M >= pair_min_tokens() && c->pair_slots > 0 && c->sm_budget == c->num_sms;
}

// Whether engram_forward over M tokens forms the gate in the projection's
// epilogue when the plan allows it (bf16 weight, whole-K tiles, shared memory
// for the fused variant).  The library's choice takes it only on CTA pairs
// (the one-CTA fused epilogue does not beat the separate gate kernel).
bool wants_fused(const engram_ctx* c, int64_t M) {
  if (c->fp8 || !gemm_can_fuse(M)) return false;
  if (c->cfg.fuse_gate >= kFuseAlways) return true;
  return c->cfg.fuse_gate == kFuseAuto && M >= fuse_auto_min_tokens() && pair_eligible(c, M);
}

constexpr int64_t kBulkEpilogueTokens = 2048;
constexpr int64_t kKeepWeightTokens = 2048;

Plan make_plan(const engram_ctx* c, int64_t M) {
  Plan p{};
  p.m_tiles = static_cast<int32_t>((M + kBM - 1) / kBM);
  p.n_tiles = c->N / kBN;
  const int32_t kbt = c->K / (c->fp8 ? 128 : kBK);
  const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
  const int64_t sms = c->sm_budget;
  auto waves = [&](int64_t units) { return (units + sms - 1) / sms; };
  int32_t best = 1;
  int64_t best_cost = waves(tiles) * kbt;
  // A small batch streams the weight at the HBM rate once at least 5/8 of the
  // SMs stream it (measured on GB300: 100 whole-K tiles on 100 of 152 SMs,
  // decode 64 tokens 56.6 -> 54.6 us for the projection, against three K
  // ranges on all 152 SMs), and without split-K the epilogue stores bf16 kv
  // and the gate reads it instead of the fp32 partial sums.  Split-K is for
  // fewer tiles than that, or more than one wave of them (an SM budget).
  const bool streams_whole = tiles <= sms && tiles * 8 >= sms * 5;
  if (M <= kSplitMaxTokens && M <= c->part_tokens && !streams_whole) {
    const int32_t cand[] = {2, 3, 4, 6, 8};
    for (int32_t s : cand) {
      if (s > kMaxSplits || kbt % s != 0) continue;
      const int64_t cost = waves(tiles * s) * (kbt / s);
      if (cost < best_cost) {
        best_cost = cost;
        best = s;
      }
    }
  }
  // tuning override for measurements: ENGRAM_SPLITS=<s> forces a split-K factor
  static const int forced = [] {
    const char* e = std::getenv("ENGRAM_SPLITS");
    return e != nullptr ? std::atoi(e) : 0;
  }();
  if (forced >= 1 && forced <= kMaxSplits && kbt % forced == 0 &&
      (forced == 1 || (M <= kSplitMaxTokens && M <= c->part_tokens)))
    best = forced;
  p.splits = best;
  p.units = tiles * best;
  // CTA pairs: each SM holds and reads half of every weight tile it
  // multiplies, so the shared memory's bandwidth, which bounds the one-CTA
  // tile, goes further.  Tiles of 256 x 256.
  if (best == 1 && pair_eligible(c, M) && !(forced >= 1 && forced <= kMaxSplits)) {
    const int64_t pair_tiles = static_cast<int64_t>((p.m_tiles + 1) / 2) * p.n_tiles;
    const int64_t slots = c->pair_slots;
    p.pair = true;
    p.units = pair_tiles;
    // a small last wave of pair tiles is cut into K ranges, as for one-CTA
    // tiles below (4,096 tokens: 1,600 tiles on 76 pairs leave 4); not with
    // the fused gate epilogue, which takes whole tiles
    const int64_t prem = pair_tiles % slots;
    if (c->rem_ws != nullptr && !wants_fused(c, M) && pair_tiles > slots && prem > 0 && prem <= slots / 4) {
      int64_t best_rem = kbt;
      for (int32_t sp = 2; sp <= kMaxRemSplits; ++sp) {
        if (kbt % sp != 0) continue;
        const int64_t cost = ((prem * sp + slots - 1) / slots) * (kbt / sp);
        if (cost < best_rem) {
          best_rem = cost;
          p.rem_splits = sp;
        }
      }
      if (p.rem_splits > 0) {
        p.rem_tiles = static_cast<int32_t>(prem);
        p.units = (pair_tiles - prem) + prem * p.rem_splits;
      }
    }
    p.ctas = static_cast<int32_t>(2 * (p.units < slots ? p.units : slots));
    return p;
  }
  // Without split-K, a last wave of rem < sms tiles would leave SMs idle for
  // a whole tile's K loop: cut those tiles into rem_splits K ranges when that
  // shortens the last wave (each range's fp32 sums go to a workspace; the last
  // range of a tile to finish adds them up in order).  A context with the
  // fused gate epilogue (for this batch size) keeps whole tiles, so that its
  // forward and its lookup_project + gate_apply sum kv in the same order.
  // Only a small last wave is cut (at most a quarter of the grid): measured on
  // GB300, 8 of 152 tiles (4096 tokens) gain 2.5 %, while 96 of 152 (512
  // tokens) lose to the cut tiles' extra epilogues and the reduction.
  const int64_t rem = tiles % sms;
  if (best == 1 && c->rem_ws != nullptr && !wants_fused(c, M) && tiles > sms && rem > 0 && rem <= sms / 4 &&
      !(forced >= 1 && forced <= kMaxSplits)) {
    int64_t best_rem = kbt;                          // cost of the partial wave as it is
    for (int32_t s = 2; s <= kMaxRemSplits; ++s) {
      if (kbt % s != 0) continue;
      const int64_t cost = waves(rem * s) * (kbt / s);
      if (cost < best_rem) {
        best_rem = cost;
        p.rem_splits = s;
      }
    }
    if (p.rem_splits > 0) {
      p.rem_tiles = static_cast<int32_t>(rem);
      p.units = (tiles - rem) + rem * p.rem_splits;
    }
  }
  p.ctas = static_cast<int32_t>(p.units < sms ? p.units : sms);
  return p;
}

engram_status check_tokens(const engram_ctx* c, int64_t B, int64_t T, int64_t* M) {
  if (B < 0 || T < 0) return ENGRAM_EINVAL;
  if (B != 0 && T > INT64_MAX / B) return ENGRAM_EINVAL;
  *M = B * T;
  if (*M > c->cfg.max_tokens) return ENGRAM_EINVAL;
  return ENGRAM_OK;
}

engram_status cuda_status(cudaError_t e) { return e == cudaSuccess ? ENGRAM_OK : ENGRAM_ECUDA; }

// Stage event i (0: before the gather, 1-3: after each stage) of the current
// call; event 3 ends the call.
void mark(engram_ctx* c, int i, cudaStream_t s) {
  if (!c->timing) return;
  cudaEventRecord(c->ev[(c->timing_calls % c->timing_sets) * 4 + i], s);
  if (i == 3) ++c->timing_calls;
}

void destroy_events(engram_ctx* c) {
  if (c->ev != nullptr) {
    for (int64_t i = 0; i < 4 * static_cast<int64_t>(c->timing_sets); ++i)
      if (c->ev[i] != nullptr) cudaEventDestroy(c->ev[i]);
    delete[] c->ev;
  }
  c->ev = nullptr;
  c->timing_sets = 0;
  c->timing_calls = 0;
  c->timing = false;
}

GatherArgs gather_args(const engram_ctx* c, const int64_t* ids, uint16_t* out, int64_t M) {
  GatherArgs g{};
  g.ids = ids;
  g.table = c->w.table;
  g.scale = c->w.scale;
  g.out = out;
  g.rows_total = M * c->cfg.n_cols;
  g.R = c->cfg.num_rows;
  g.row0 = c->cfg.row_offset;
  g.head_dim = c->cfg.head_dim;
  g.scale_block = c->cfg.scale_block;
  g.scale_fmt = c->cfg.scale_fmt;
  g.check_ids = c->cfg.check_ids;
  g.err = c->err;
  return g;
}

// The hidden-state side of engram_forward: with it, a plan without split-K runs
// the gate and the residual add in the projection's epilogue.
struct FusedIO {
  const uint16_t* x;
  const uint8_t* mask;
  uint16_t* out;
};

bool fuses(const engram_ctx* c, const Plan& p, int64_t M) { return p.splits == 1 && wants_fused(c, M); }

// gathered rows -> projection.  The rows are gathered from `ids` into the
// context's buffer, or, with rows_in (bf16 weight only), taken from the
// caller.  With `fused` and a fusable plan it writes the layer's output;
// otherwise bf16 kv to kv_out when splits == 1 and the fp32 partial sums to
// the context when splits > 1.
engram_status run_projection(engram_ctx* c, const int64_t* ids, const uint16_t* rows_in, int64_t M, uint16_t* kv_out,
                             const FusedIO* fused, Plan* plan_out, cudaStream_t stream) {
  if (cudaSetDevice(c->device) != cudaSuccess) return ENGRAM_ECUDA;
  const Plan p = make_plan(c, M);
  const bool fuse = fused != nullptr && fuses(c, p, M);
  GatherArgs g = gather_args(c, ids, c->rows, M);
  const bool rem = !fuse && p.rem_splits > 0;
  if (fuse) {
    g.zero = c->counters;
    g.n_zero = p.m_tiles * 8;
  }
  mark(c, 0, stream);
  if (rows_in != nullptr) {
    // no gather: clear what it would have cleared for the fused epilogue
    if (fuse && cudaMemsetAsync(c->counters, 0, static_cast<size_t>(p.m_tiles) * 8 * sizeof(uint32_t), stream) !=
                    cudaSuccess)
      return ENGRAM_ECUDA;
  } else if (c->fp8) {
    if (launch_gather_codes(g, c->cfg.n_cols, c->codes, c->sfa, c->num_sms, stream) != cudaSuccess)
      return ENGRAM_ECUDA;
  } else if (launch_gather(g, c->num_sms, stream) != cudaSuccess) {
    return ENGRAM_ECUDA;
  }
  mark(c, 1, stream);
  GemmArgs a{};
  a.M = M;
  a.N = c->N;
  a.K = c->K;
  a.splits = p.splits;
  a.kb_per_split = (c->K / (c->fp8 ? 128 : kBK)) / p.splits;
  a.m_tiles = p.m_tiles;
  a.n_tiles = p.n_tiles;
  a.group_m = p.m_tiles < 16 ? p.m_tiles : 16;
  if (p.pair) {
    const int32_t m_pairs = (p.m_tiles + 1) / 2;
    a.pair = 1;
    a.group_m = m_pairs < 8 ? m_pairs : 8;       // 8 pairs = the same 16 M tiles per group
  }
  a.units = p.units;
  a.full_units = static_cast<int64_t>(p.m_tiles) * p.n_tiles * p.splits;
  if (rem) {
    a.full_units = (p.pair ? static_cast<int64_t>((p.m_tiles + 1) / 2) : p.m_tiles) * p.n_tiles - p.rem_tiles;
    a.rem_tiles = p.rem_tiles;
    a.rem_splits = p.rem_splits;
    a.rem_kb = (c->K / (c->fp8 ? 128 : kBK)) / p.rem_splits;
    a.rem_ws = c->rem_ws;
  }
  a.out_mode = p.splits == 1 ? kOutBf16 : kOutPartial;
  a.kv = kv_out;
  a.part = c->part;
  a.err = c->err;
  a.wpack = c->wpack;
  // per-row bulk-copy stores in the epilogue pay off once a bf16 batch is large
  // (4,096 tokens: 911 -> 887 us, 16,384: 4.04 -> 3.81 ms) and cost while the
  // weight streams (decode, 512 tokens) or in the MXFP8 kernel (4,096 tokens:
  // 614 -> 757 us), where the copies queue with the many small scale loads
  a.bulk_epilogue = !c->fp8 && M >= kBulkEpilogueTokens ? 1 : 0;
  // a weight tile is read by every M tile of a 16-tile group; from 16 M tiles
  // on, those reads drift apart in time and an evict-first tile is often gone
  // before the last of them (measured on GB300, evict-last: 4,096 tokens
  // 886 -> 857 us, MXFP8 610 -> 587 us, 16,384 tokens 3.77 -> 3.50 ms; at 512
  // tokens, 4 M tiles in step, it cost 134 -> 140 us)
  a.keep_weight = M >= kKeepWeightTokens ? 1 : 0;
  a.fp8 = c->fp8 ? 1 : 0;
  a.sfa = c->sfa;
  a.sfb = c->wsf;
  if (fuse) {
    a.out_mode = kOutFused;
    a.x = fused->x;
    a.mask = fused->mask;
    a.wprod = c->wprod;
    a.out = fused->out;
    a.gsum = c->gsum;
    a.counters = c->counters;
    a.tickets = c->tickets;
    a.gates = c->gates;
    a.key_n_tiles = c->cfg.hc_mult * c->cfg.dim / kBN;
    a.hold_ready_flags = (c->test_hooks & ENGRAM_TEST_HOLD_GATE_FLAGS) != 0 ? 1 : 0;
    a.dim = c->cfg.dim;
    a.hc = c->cfg.hc_mult;
    a.eps = c->cfg.eps;
    a.clamp = c->cfg.clamp;
    a.inv_sqrt_dim = static_cast<float>(1.0 / std::sqrt(static_cast<double>(c->cfg.dim)));
  }
  const void* rows = rows_in != nullptr ? static_cast<const void*>(rows_in)
                     : c->fp8        ? static_cast<const void*>(c->codes)
                                     : static_cast<const void*>(c->rows);
  if (launch_gemm(rows, c->tmW, a, p.ctas, stream) != cudaSuccess) return ENGRAM_ECUDA;
  if (rem && launch_reduce_remainder(a, c->num_sms, stream) != cudaSuccess) return ENGRAM_ECUDA;
  mark(c, 2, stream);
  *plan_out = p;
  return ENGRAM_OK;
}

GateArgs gate_args(const engram_ctx* c, const uint16_t* x, const uint8_t* mask, uint16_t* out, float* gates,
                   int64_t M) {
  GateArgs a{};
  a.x = x;
  a.mask = mask;
  a.wprod = c->wprod;
  a.out = out;
  a.gates = gates;
  a.M = M;
  a.dim = c->cfg.dim;
  a.hc = c->cfg.hc_mult;
  a.eps = c->cfg.eps;
  a.clamp = c->cfg.clamp;
  a.inv_sqrt_dim = static_cast<float>(1.0 / std::sqrt(static_cast<double>(c->cfg.dim)));
  a.err = c->err;
  a.num_sms = c->num_sms;
  return a;
}

void free_ctx(engram_ctx* c) {
  if (c == nullptr) return;
  destroy_events(c);
  cudaFree(c->wprod);
  cudaFree(c->rows);
  cudaFree(c->kv);
  cudaFree(c->part);
  cudaFree(c->err);
  cudaFree(c->gsum);
  cudaFree(c->counters);
  cudaFree(c->tickets);
  cudaFree(c->gates);
  cudaFree(c->wpack);
  cudaFree(c->rem_ws);
  cudaFree(c->wsf);
  cudaFree(c->codes);
  cudaFree(c->sfa);
  delete c;
}

// The layer from ids (gathered here) or from caller rows: projection, then the
// gate in the projection's epilogue or in the gate kernel.
engram_status forward_from(engram_ctx* ctx, const int64_t* hash_ids, const uint16_t* rows, const uint16_t* x,
                           const uint8_t* token_mask, uint16_t* out, int64_t M, cudaStream_t s) {
  Plan p{};
  const FusedIO io{x, token_mask, out};
  engram_status st = run_projection(ctx, hash_ids, rows, M, ctx->kv, &io, &p, s);
  if (st != ENGRAM_OK) return st;
  if (fuses(ctx, p, M)) {   // the projection's epilogue applied the gate
    mark(ctx, 3, s);
    return ENGRAM_OK;
  }
  GateArgs g = gate_args(ctx, x, token_mask, out, nullptr, M);
  if (p.splits == 1) {
    g.kv = ctx->kv;
  } else {
    g.part = ctx->part;
    g.splits = p.splits;
  }
  st = cuda_status(launch_gate(g, s));
  mark(ctx, 3, s);
  return st;
}

}  // namespace

extern "C" {

const char* engram_status_string(engram_status s) {
  switch (s) {
    case ENGRAM_OK: return "ok";
    case ENGRAM_EINVAL: return "invalid argument";
    case ENGRAM_ENOMEM: return "out of memory";
    case ENGRAM_ECUDA: return "CUDA error";
    case ENGRAM_ERANGE: return "hash id outside the table";
    case ENGRAM_ETIMEOUT: return "kernel wait timed out";
    case ENGRAM_EUNSUPPORTED: return "unsupported shape or format";
  }
  return "unknown status";
}

int32_t engram_abi_version(void) { return 105; }

engram_status engram_create(engram_ctx** out, const engram_config* cfg, const engram_weights* w) {
  if (out == nullptr || cfg == nullptr || w == nullptr) return ENGRAM_EINVAL;
  *out = nullptr;
  const engram_config& c = *cfg;
  if (c.dim <= 0 || c.hc_mult <= 0 || c.n_cols <= 0 || c.head_dim <= 0 || c.scale_block <= 0 ||
      c.num_rows < 0 || c.max_tokens < 0 || !(c.eps >= 0.0f) || !(c.clamp >= 0.0f) || c.row_offset < 0 ||
      c.row_offset > INT64_MAX - c.num_rows)
    return ENGRAM_EINVAL;
  if (w->table == nullptr || w->scale == nullptr || w->wkv == nullptr || w->q_weight == nullptr ||
      w->k_weight == nullptr)
    return ENGRAM_EINVAL;
  if (!aligned(w->table, 16) || !aligned(w->wkv, 16) || !aligned(w->q_weight, 16) || !aligned(w->k_weight, 16) ||
      !aligned(w->scale, c.scale_fmt == ENGRAM_SCALE_F32 ? 4 : 1))
    return ENGRAM_EINVAL;
  if (c.scale_fmt != ENGRAM_SCALE_F32 && c.scale_fmt != ENGRAM_SCALE_E8M0) return ENGRAM_EUNSUPPORTED;
  if (c.dim % kBN != 0 || c.dim > 5120 || c.hc_mult > 4) return ENGRAM_EUNSUPPORTED;
  if (c.head_dim % 16 != 0 || c.head_dim % c.scale_block != 0 || c.scale_block % 16 != 0)
    return ENGRAM_EUNSUPPORTED;
  const int64_t K = static_cast<int64_t>(c.n_cols) * c.head_dim;
  const int64_t N = static_cast<int64_t>(c.dim) * (c.hc_mult + 1);
  if (K % kBK != 0 || K > (1 << 20) || N > (1 << 24)) return ENGRAM_EUNSUPPORTED;
  if (c.wkv_fmt != ENGRAM_WKV_BF16 && c.wkv_fmt != ENGRAM_WKV_MXFP8) return ENGRAM_EUNSUPPORTED;
  const bool fp8 = c.wkv_fmt == ENGRAM_WKV_MXFP8;
  if (fp8) {
    // the table's codes and scales feed the block-scaled MMA as they are
    if (c.scale_fmt != ENGRAM_SCALE_E8M0 || c.scale_block != 32 || K % 128 != 0) return ENGRAM_EUNSUPPORTED;
    if (w->wkv_scale == nullptr) return ENGRAM_EINVAL;
  }

  engram_ctx* ctx = new (std::nothrow) engram_ctx();
  if (ctx == nullptr) return ENGRAM_ENOMEM;
  ctx->cfg = c;
  ctx->w = *w;
  ctx->K = static_cast<int32_t>(K);
  ctx->N = static_cast<int32_t>(N);
  ctx->fp8 = fp8;
  if (cudaGetDevice(&ctx->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device) != cudaSuccess) {
    delete ctx;
    return ENGRAM_ECUDA;
  }
  if (!device_readable(w->table, ctx->device) || !device_readable(w->scale, ctx->device) ||
      !device_readable(w->wkv, ctx->device) || !device_readable(w->q_weight, ctx->device) ||
      !device_readable(w->k_weight, ctx->device) || (fp8 && !device_readable(w->wkv_scale, ctx->device))) {
    delete ctx;
    return ENGRAM_EINVAL;
  }
  int cc_major = 0, cc_minor = 0;
  cudaDeviceGetAttribute(&cc_major, cudaDevAttrComputeCapabilityMajor, ctx->device);
  cudaDeviceGetAttribute(&cc_minor, cudaDevAttrComputeCapabilityMinor, ctx->device);
  if (cc_major != 10 || cc_minor != 3) {   // sm_103a code only
    delete ctx;
    return ENGRAM_EUNSUPPORTED;
  }
  ctx->sm_budget = ctx->num_sms;
  ctx->pair_slots = 0;
  const int64_t mt = c.max_tokens > 0 ? c.max_tokens : 1;
  ctx->part_tokens = mt < kSplitMaxTokens ? mt : kSplitMaxTokens;
  const size_t hcd = static_cast<size_t>(c.hc_mult) * c.dim;
  bool ok = cudaMalloc(&ctx->wprod, hcd * sizeof(float)) == cudaSuccess &&
            cudaMalloc(&ctx->rows, static_cast<size_t>(mt) * K * 2) == cudaSuccess &&
            cudaMalloc(&ctx->kv, static_cast<size_t>(mt) * N * 2) == cudaSuccess &&
            cudaMalloc(&ctx->part, static_cast<size_t>(kMaxSplits) * ctx->part_tokens * N * 4) == cudaSuccess &&
            cudaMalloc(&ctx->err, 2 * sizeof(unsigned long long)) == cudaSuccess &&
            cudaMalloc(&ctx->gsum, static_cast<size_t>(mt) * c.hc_mult * (c.dim / kBN) * 4 * sizeof(float)) ==
                cudaSuccess &&
            cudaMalloc(&ctx->counters, static_cast<size_t>((mt + kBM - 1) / kBM) * 8 * sizeof(uint32_t)) ==
                cudaSuccess &&
            cudaMalloc(&ctx->gates, static_cast<size_t>(mt) * 4 * sizeof(float)) == cudaSuccess &&
            cudaMalloc(&ctx->tickets, 2 * sizeof(uint32_t)) == cudaSuccess &&
            cudaMalloc(&ctx->wpack, static_cast<size_t>(N) * K * (fp8 ? 1 : 2)) == cudaSuccess;
  const size_t sfa_bytes = static_cast<size_t>((mt + kBM - 1) / kBM) * (K / 128) * 512;
  if (ok && mt > kSplitMaxTokens)
    ok = cudaMalloc(&ctx->rem_ws, static_cast<size_t>(ctx->num_sms) * kMaxRemSplits * kBM * kBN * sizeof(float)) ==
         cudaSuccess;
  if (ok && fp8)
    ok = cudaMalloc(&ctx->wsf, static_cast<size_t>(N) * (K / 32)) == cudaSuccess &&
         cudaMalloc(&ctx->codes, static_cast<size_t>(mt) * K) == cudaSuccess &&
         cudaMalloc(&ctx->sfa, sfa_bytes) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    free_ctx(ctx);
    return ENGRAM_ENOMEM;
  }
  if (cudaMemset(ctx->err, 0, 2 * sizeof(unsigned long long)) != cudaSuccess ||
      cudaMemset(ctx->tickets, 0, 2 * sizeof(uint32_t)) != cudaSuccess ||
      launch_weight_product(w->q_weight, w->k_weight, ctx->wprod, static_cast<int64_t>(hcd), nullptr) !=
          cudaSuccess ||
      (fp8 ? launch_pack_wkv(static_cast<const uint16_t*>(w->wkv), N, K / 2, ctx->wpack, nullptr) != cudaSuccess ||
                 launch_pack_sfb(w->wkv_scale, N, K, ctx->wsf, nullptr) != cudaSuccess ||
                 cudaMemset(ctx->sfa, 127, sfa_bytes) != cudaSuccess   // scales of rows past M: 1.0
           : launch_pack_wkv(static_cast<const uint16_t*>(w->wkv), N, K, ctx->wpack, nullptr) != cudaSuccess) ||
      gemm_prepare() != cudaSuccess || gate_prepare() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    free_ctx(ctx);
    return ENGRAM_ECUDA;
  }
  ctx->pair_slots = gemm_pair_slots(ctx->num_sms);
  if (!fp8 && !make_tmap_bf16(&ctx->tmW, w->wkv, static_cast<uint64_t>(N), static_cast<uint64_t>(K), kBN)) {
    free_ctx(ctx);
    return ENGRAM_ECUDA;
  }
  *out = ctx;
  return ENGRAM_OK;
}

void engram_destroy(engram_ctx* ctx) {
  if (ctx == nullptr) return;
  cudaSetDevice(ctx->device);
  cudaDeviceSynchronize();
  free_ctx(ctx);
}

engram_status engram_forward(engram_ctx* ctx, const int64_t* hash_ids, const uint16_t* x,
                             const uint8_t* token_mask, uint16_t* out, int64_t B, int64_t T,
                             engram_stream_t stream) {
  if (ctx == nullptr) return ENGRAM_EINVAL;
  int64_t M;
  engram_status st = check_tokens(ctx, B, T, &M);
  if (st != ENGRAM_OK) return st;
  if (M == 0) return ENGRAM_OK;
  if (hash_ids == nullptr || x == nullptr || out == nullptr) return ENGRAM_EINVAL;
  if (!aligned(hash_ids, 8) || !aligned(x, 16) || !aligned(out, 16)) return ENGRAM_EINVAL;
  return forward_from(ctx, hash_ids, nullptr, x, token_mask, out, M, reinterpret_cast<cudaStream_t>(stream));
}

engram_status engram_forward_rows(engram_ctx* ctx, const uint16_t* rows, const uint16_t* x,
                                  const uint8_t* token_mask, uint16_t* out, int64_t B, int64_t T,
                                  engram_stream_t stream) {
  if (ctx == nullptr) return ENGRAM_EINVAL;
  if (ctx->fp8) return ENGRAM_EUNSUPPORTED;   // the MXFP8 projection reads the table's codes, not bf16 rows
  int64_t M;
  engram_status st = check_tokens(ctx, B, T, &M);
  if (st != ENGRAM_OK) return st;
  if (M == 0) return ENGRAM_OK;
  if (rows == nullptr || x == nullptr || out == nullptr) return ENGRAM_EINVAL;
  if (!aligned(rows, 16) || !aligned(x, 16) || !aligned(out, 16)) return ENGRAM_EINVAL;
  return forward_from(ctx, nullptr, rows, x, token_mask, out, M, reinterpret_cast<cudaStream_t>(stream));
}

engram_status engram_lookup_project(engram_ctx* ctx, const int64_t* hash_ids, uint16_t* kv, int64_t B,
                                    int64_t T, engram_stream_t stream) {
  if (ctx == nullptr) return ENGRAM_EINVAL;
  int64_t M;
  engram_status st = check_tokens(ctx, B, T, &M);
  if (st != ENGRAM_OK) return st;
  if (M == 0) return ENGRAM_OK;
  if (hash_ids == nullptr || kv == nullptr || !aligned(hash_ids, 8) || !aligned(kv, 16)) return ENGRAM_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Plan p{};
  st = run_projection(ctx, hash_ids, nullptr, M, kv, nullptr, &p, s);
  if (st != ENGRAM_OK) return st;
  if (p.splits > 1) st = cuda_status(launch_reduce_partials(ctx->part, p.splits, M, ctx->N, kv, ctx->num_sms, s));
  mark(ctx, 3, s);
  return st;
}

engram_status engram_gate_apply(engram_ctx* ctx, const uint16_t* kv, const uint16_t* x, const uint8_t* token_mask,
                                uint16_t* out, float* gates, int64_t B, int64_t T, engram_stream_t stream) {
  if (ctx == nullptr) return ENGRAM_EINVAL;
  int64_t M;
  engram_status st = check_tokens(ctx, B, T, &M);
  if (st != ENGRAM_OK) return st;
  if (M == 0) return ENGRAM_OK;
  if (kv == nullptr || x == nullptr || out == nullptr) return ENGRAM_EINVAL;
  if (!aligned(kv, 16) || !aligned(x, 16) || !aligned(out, 16) || !aligned(gates, 4)) return ENGRAM_EINVAL;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return ENGRAM_ECUDA;
  GateArgs g = gate_args(ctx, x, token_mask, out, gates, M);
  g.kv = kv;
  return cuda_status(launch_gate(g, reinterpret_cast<cudaStream_t>(stream)));
}

engram_status engram_lookup(engram_ctx* ctx, const int64_t* hash_ids, uint16_t* rows, int64_t B, int64_t T,
                            engram_stream_t stream) {
  if (ctx == nullptr) return ENGRAM_EINVAL;
  int64_t M;
  engram_status st = check_tokens(ctx, B, T, &M);
  if (st != ENGRAM_OK) return st;
  if (M == 0) return ENGRAM_OK;
  if (hash_ids == nullptr || rows == nullptr || !aligned(hash_ids, 8) || !aligned(rows, 16)) return ENGRAM_EINVAL;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return ENGRAM_ECUDA;
  GatherArgs g = gather_args(ctx, hash_ids, rows, M);
  return cuda_status(launch_gather(g, ctx->num_sms, reinterpret_cast<cudaStream_t>(stream)));
}

engram_status engram_sync_status(engram_ctx* ctx, engram_stream_t stream, int64_t* bad_ids) {
  if (ctx == nullptr) return ENGRAM_EINVAL;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return ENGRAM_ECUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned long long h[2] = {0, 0};
  if (cudaStreamSynchronize(s) != cudaSuccess) return ENGRAM_ECUDA;
  if (cudaMemcpy(h, ctx->err, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return ENGRAM_ECUDA;
  if (cudaMemset(ctx->err, 0, sizeof(h)) != cudaSuccess) return ENGRAM_ECUDA;
  if (bad_ids != nullptr) *bad_ids = static_cast<int64_t>(h[1]);
  if (h[0] & kErrTimeout) return ENGRAM_ETIMEOUT;
  if (h[0] & kErrRange) return ENGRAM_ERANGE;
  return ENGRAM_OK;
}

engram_status engram_enable_stage_timing(engram_ctx* ctx, int32_t enable) {
  if (ctx == nullptr || enable < 0 || enable > kMaxTimedCalls) return ENGRAM_EINVAL;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return ENGRAM_ECUDA;
  destroy_events(ctx);
  if (enable == 0) return ENGRAM_OK;
  ctx->ev = new (std::nothrow) cudaEvent_t[4 * static_cast<size_t>(enable)]();
  if (ctx->ev == nullptr) return ENGRAM_ENOMEM;
  ctx->timing_sets = enable;
  for (int64_t i = 0; i < 4 * static_cast<int64_t>(enable); ++i) {
    if (cudaEventCreate(&ctx->ev[i]) != cudaSuccess) {
      destroy_events(ctx);
      return ENGRAM_ECUDA;
    }
  }
  ctx->timing = true;
  return ENGRAM_OK;
}

engram_status engram_stage_times_n(engram_ctx* ctx, int32_t n, float* ms) {
  if (ctx == nullptr || ms == nullptr || !ctx->timing || n < 1 || n > ctx->timing_sets ||
      n > ctx->timing_calls)
    return ENGRAM_EINVAL;
  const int64_t last = ctx->timing_calls - 1;
  if (cudaEventSynchronize(ctx->ev[(last % ctx->timing_sets) * 4 + 3]) != cudaSuccess) return ENGRAM_ECUDA;
  for (int32_t k = 0; k < n; ++k) {
    const cudaEvent_t* e = ctx->ev + ((last - (n - 1) + k) % ctx->timing_sets) * 4;
    for (int i = 0; i < 3; ++i)
      if (cudaEventElapsedTime(&ms[3 * k + i], e[i], e[i + 1]) != cudaSuccess) return ENGRAM_ECUDA;
  }
  return ENGRAM_OK;
}

engram_status engram_stage_times(engram_ctx* ctx, float* ms) { return engram_stage_times_n(ctx, 1, ms); }

engram_status engram_test_hook(engram_ctx* ctx, int32_t hooks) {
  if (ctx == nullptr || (hooks & ~ENGRAM_TEST_HOLD_GATE_FLAGS) != 0) return ENGRAM_EINVAL;
  ctx->test_hooks = hooks;
  return ENGRAM_OK;
}

engram_status engram_set_sm_budget(engram_ctx* ctx, int32_t sms) {
  if (ctx == nullptr || sms < 0) return ENGRAM_EINVAL;
  ctx->sm_budget = (sms == 0 || sms > ctx->num_sms) ? ctx->num_sms : sms;
  return ENGRAM_OK;
}

engram_status engram_plan(const engram_ctx* ctx, int64_t m_tokens, int32_t* splits, int32_t* ctas) {
  if (ctx == nullptr || m_tokens < 0) return ENGRAM_EINVAL;
  const Plan p = make_plan(ctx, m_tokens);
  if (splits != nullptr) *splits = p.splits;
  if (ctas != nullptr) *ctas = p.ctas;
  return ENGRAM_OK;
}

engram_status engram_describe_plan(const engram_ctx* ctx, int64_t m_tokens, engram_plan_info* info) {
  if (ctx == nullptr || m_tokens < 0 || info == nullptr) return ENGRAM_EINVAL;
  const Plan p = make_plan(ctx, m_tokens);
  info->splits = p.splits;
  info->ctas = p.ctas;
  info->cta_pairs = p.pair ? 1 : 0;
  info->rem_tiles = p.rem_tiles;
  info->rem_splits = p.rem_splits;
  info->fused_gate = m_tokens > 0 && fuses(ctx, p, m_tokens) ? 1 : 0;
  return ENGRAM_OK;
}

engram_status engram_forward_kernels(const engram_ctx* ctx, int64_t m_tokens, int32_t* kernels) {
  if (ctx == nullptr || m_tokens < 0 || kernels == nullptr) return ENGRAM_EINVAL;
  if (m_tokens == 0) {
    *kernels = 0;
    return ENGRAM_OK;
  }
  const Plan p = make_plan(ctx, m_tokens);
  if (fuses(ctx, p, m_tokens)) {
    *kernels = 2;                                   // gather, projection with the gate in its epilogue
  } else {
    *kernels = 3 + (p.rem_splits > 0 ? 1 : 0);      // gather, projection, [remainder sums], gate
  }
  return ENGRAM_OK;
}

}  // extern "C"
