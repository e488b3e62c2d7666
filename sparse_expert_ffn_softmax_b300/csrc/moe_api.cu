// C ABI of the library: argument validation, workspace layout and the stage
// entry points declared in include/moe.h. Every step of the layer runs in the
// kernels of router.cu, permute.cu, ffn_simt.cu and gemm_tc.cu; this file only
// checks arguments, carves the caller's workspace and enqueues launches.
#include <cmath>
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "stats.cuh"

namespace moe {
namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }
inline bool ok_opt(const void* p) { return p == nullptr || aligned16(p); }

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace

moe_status make_plan(const moe_config* c, Plan* p) {
  if (!c || !p) return MOE_ERR_INVALID_ARG;
  std::memset(p, 0, sizeof(*p));
  p->cfg = *c;
  p->N = c->n_tokens;
  p->d = c->d_model;
  p->F = c->d_ff;
  p->E = c->n_experts;
  p->S = c->n_shared;
  p->Fs = c->d_ff_shared;
  p->k = c->top_k;
  if (p->N < 0 || p->d < 1 || p->F < 1 || p->E < 1 || p->k < 1 || p->S < 0) return MOE_ERR_INVALID_ARG;
  if (p->S > 0 && p->Fs < 1) return MOE_ERR_INVALID_ARG;
  if (c->gating < 0 || c->gating > 3 || c->act < 0 || c->act > 1 || c->dtype < 0 || c->dtype > 1)
    return MOE_ERR_INVALID_ARG;
  if (!std::isfinite(c->capacity_factor) || !std::isfinite(c->aux_alpha)) return MOE_ERR_INVALID_ARG;
  if (c->n_tokens_total != 0 && c->n_tokens_total < c->n_tokens) return MOE_ERR_INVALID_ARG;
  if ((c->flags & ~(int32_t)(MOE_FLAG_DROP_PASSTHROUGH | MOE_FLAG_GATHER_ROWS)) != 0) return MOE_ERR_INVALID_ARG;
  if (c->weight_format != MOE_WEIGHTS_DTYPE && c->weight_format != MOE_WEIGHTS_MXFP8) return MOE_ERR_INVALID_ARG;
  p->Ntot = c->n_tokens_total > p->N ? c->n_tokens_total : p->N;
  p->sharded = p->Ntot > p->N;
  p->passthrough = (c->flags & MOE_FLAG_DROP_PASSTHROUGH) != 0;
  if (p->k > p->E || p->k > 32 || p->E > 512 || p->S > 64) return MOE_ERR_UNSUPPORTED;
  p->bf16 = c->dtype == MOE_DT_BF16;
  p->gather = p->bf16 && (c->flags & MOE_FLAG_GATHER_ROWS) != 0;
  p->fp8w = c->weight_format == MOE_WEIGHTS_MXFP8;
  if (p->fp8w && (!p->bf16 || p->gather || p->d % 512 || p->F % 512)) return MOE_ERR_UNSUPPORTED;
  p->swiglu = c->act == MOE_ACT_SWIGLU;
  p->ec = c->gating == MOE_GATE_EXPERT_CHOICE;
  p->bias = c->has_bias != 0;
  if (p->swiglu && p->bias) return MOE_ERR_UNSUPPORTED;
  if (p->bf16) {
    if (p->d % 64 || p->F % 64 || (p->S > 0 && p->Fs % 64)) return MOE_ERR_UNSUPPORTED;
  } else {
    if (p->d % 4) return MOE_ERR_UNSUPPORTED;
  }
  if (p->N * p->k >= (int64_t)1 << 31) return MOE_ERR_UNSUPPORTED;
  if (p->ec && p->N > ((int64_t)1 << 20)) return MOE_ERR_UNSUPPORTED;
  // expert choice ranks every token of the batch for every expert: a shard cannot
  // select without the other shards' candidates
  if (p->ec && p->sharded) return MOE_ERR_UNSUPPORTED;
  if (p->Ntot * p->k >= (int64_t)1 << 31) return MOE_ERR_UNSUPPORTED;
  // capacity of the whole batch: token choice C = ceil(N*k*cf/E) (cf <= 0: no limit);
  // expert choice C = min(N, ceil(N*k*cf/E)) with cf <= 0 read as 1.
  const double cf = (double)c->capacity_factor;
  if (p->ec) {
    const double cfe = cf > 0 ? cf : 1.0;
    int64_t cap = (int64_t)std::ceil((double)p->N * (double)p->k * cfe / (double)p->E);
    p->cap = cap < p->N ? cap : p->N;
  } else if (cf <= 0) {
    p->cap = p->Ntot;
  } else {
    int64_t cap = (int64_t)std::ceil((double)p->Ntot * (double)p->k * cf / (double)p->E);
    p->cap = cap < p->Ntot ? cap : p->Ntot;
  }
  if (p->cap < 0) p->cap = 0;
  p->max_rows = p->ec ? p->E * p->cap : p->N * p->k;
  if (p->max_rows >= (int64_t)1 << 31) return MOE_ERR_UNSUPPORTED;
  // smaller tiles for smaller batches, so routing and permuting still spread over the SMs.
  // A shard takes the whole batch's choices (tile, K split of the router), so its per-token
  // arithmetic and its statistic partials are those of the unsharded batch.
  p->tile = p->Ntot >= 16384 ? 32 : (p->Ntot >= 4096 ? 16 : 8);
  p->tiles = ceil_div(p->N, p->tile);
  p->words = ceil_div(p->E, 32);

  const size_t b = p->bf16 ? 2 : 4;
  const int64_t nsel = p->ec ? p->E * p->cap : p->N * p->k;
  moe_workspace_layout& L = p->L;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align_up(bytes > 0 ? bytes : 1);
    return at;
  };
  L.status = take(32);  // int32 error word [4] + last-block ticket
  L.logits = take((size_t)(p->N * p->E) * 4);
  L.probs = take((size_t)(p->N * p->E) * 4);
  L.idx = take((size_t)nsel * 4);
  L.gate = take((size_t)nsel * 4);
  L.tok_rows = take((size_t)nsel * 4);
  L.tok_off = take((size_t)(p->N + 1) * 4);
  L.expert_off = take((size_t)(p->E + 1) * 4);
  L.row_token = take((size_t)p->max_rows * 4);
  L.row_gate = take((size_t)p->max_rows * 4);
  // with MOE_FLAG_GATHER_ROWS the up-projection gathers its rows straight from x and
  // the forward writes no xp
  L.xp = take(p->gather ? 0 : (size_t)p->max_rows * (size_t)p->d * b);
  L.h = take((size_t)p->max_rows * (size_t)p->F * b);
  L.hs = take((size_t)p->N * (size_t)(p->S * p->Fs) * b);
  L.yp = take((size_t)p->max_rows * (size_t)p->d * 4);  // fp32 for every layer dtype
  L.ys = take(p->S > 0 ? (size_t)p->N * (size_t)p->d * 4 : 0);
  L.stats = take(moe_stats_bytes(p->E));
  p->stat_acc = take(stats_acc_bytes(p->E));  // zeroed by moe_workspace_init, reset by each finaliser
  L.stat_acc = p->stat_acc;
  L.scratch = o;
  p->rank_base = take((size_t)p->E * 4);
  p->tile_counts = take((size_t)(p->E * p->tiles) * 4);
  p->tile_base = take((size_t)(p->E * (p->tiles + 1)) * 4);
  p->ec_bits = take((size_t)(p->N * p->words) * 4);
  p->probs_t = take(p->ec ? (size_t)(p->N * p->E) * 4 : 0);  // expert-major probabilities
  p->rsplit = p->bf16 ? router_k_splits(p->Ntot, p->d, p->E) : 1;
  p->logits_part = take(p->rsplit > 1 ? (size_t)(p->rsplit * p->N * p->E) * 4 : 0);
  L.total_bytes = o;
  L.max_rows = p->max_rows;
  L.capacity = p->cap;
  return MOE_OK;
}

int64_t router_k_splits(int64_t N, int64_t d, int64_t E) {
  constexpr int64_t kSms = 148, kBM = 128, kBK = 64, kMinBlocks = 4;
  const int64_t kb = d / kBK, mt = (N + kBM - 1) / kBM;
  if (N <= 0 || kb <= 0 || E < kRouterTcMinE || mt >= kRouterSplitMaxTiles) return 1;
  int64_t s = kSms / mt;
  if (s > kb / kMinBlocks) s = kb / kMinBlocks;
  while (s > 1 && kb % s) --s;  // equal K ranges
  return s > 1 ? s : 1;
}

namespace {

moe_status check_ws(const Plan& p, const void* ws, size_t ws_bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < p.L.total_bytes) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

moe_status check_weights(const Plan& p, const moe_weights* w, bool router, bool experts) {
  if (!w) return MOE_ERR_INVALID_ARG;
  if (router) {
    if (!ok_ptr(w->w_router) || !ok_opt(w->logit_bias)) return MOE_ERR_INVALID_ARG;
  }
  if (experts) {
    if (!ok_ptr(w->w1) || !ok_ptr(w->w2)) return MOE_ERR_INVALID_ARG;
    if (p.swiglu && !ok_ptr(w->w3)) return MOE_ERR_INVALID_ARG;
    if (p.fp8w && (!ok_ptr(w->w1_scale) || !ok_ptr(w->w2_scale) || (p.swiglu && !ok_ptr(w->w3_scale))))
      return MOE_ERR_INVALID_ARG;
    if (p.bias && (!ok_ptr(w->b1) || !ok_ptr(w->b2))) return MOE_ERR_INVALID_ARG;
    if (p.S > 0) {
      if (!ok_ptr(w->ws1) || !ok_ptr(w->ws2)) return MOE_ERR_INVALID_ARG;
      if (p.swiglu && !ok_ptr(w->ws3)) return MOE_ERR_INVALID_ARG;
      if (p.bias && (!ok_ptr(w->bs1) || !ok_ptr(w->bs2))) return MOE_ERR_INVALID_ARG;
    }
  }
  return MOE_OK;
}

void* stats_or_ws(const Plan& p, void* stats, void* ws) { return stats ? stats : ws_at<uint8_t>(ws, p.L.stats); }

// tile_counts non-null (token choice inside moe_forward): the router also writes
// the permute's per-tile counts and a later kernel reduces the statistics.
// Otherwise (stand-alone routing, expert choice) the router finalises them.
moe_status do_route(const Plan& p, const void* x, const moe_weights* w, int32_t* idx, float* gate, float* logits,
                    float* probs, void* stats, void* ws, cudaStream_t st, int32_t* tile_counts = nullptr) {
  float* pr = probs;
  if (p.ec && !pr) pr = ws_at<float>(ws, p.L.probs);
  cudaError_t e = launch_router(p, x, w, idx, gate, logits, pr, stats_or_ws(p, stats, ws), ws, st, tile_counts,
                                tile_counts == nullptr);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (p.ec) {
    e = launch_ec_select(p, pr, idx, gate, ws_at<float>(ws, p.probs_t), st);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status do_ffn(const Plan& p, const void* xp, const int32_t* expert_off, const float* row_gate, const void* x,
                  const moe_weights* w, void* yp, void* ys, void* ws, cudaStream_t st, int part,
                  const int32_t* gather_rows = nullptr, int families = kRoutedFamily | kSharedFamily) {
  void* h = ws_at<uint8_t>(ws, p.L.h);
  void* hs = ws_at<uint8_t>(ws, p.L.hs);
  cudaError_t e = p.bf16 ? launch_ffn_bf16(p, xp, expert_off, row_gate, x, w, h, hs, yp, ys, status_ptr(p, ws), st,
                                           part, gather_rows, families)
                         : launch_ffn_f32(p, xp, expert_off, row_gate, x, w, h, hs, yp, ys, status_ptr(p, ws), st,
                                          part);
  return cuda_status(e);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported layer shape";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_CHECK: return "device-side index check failed";
    case MOE_ERR_TIMEOUT: return "device-side pipeline wait timed out";
  }
  return "unknown status";
}

size_t moe_stat_acc_bytes(int64_t n_experts) { return stats_acc_bytes(n_experts < 0 ? 0 : n_experts); }

size_t moe_stats_bytes(int64_t n_experts) {
  if (n_experts < 0) n_experts = 0;
  return sizeof(moe_stats_header) + (size_t)n_experts * 16;
}

moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  Plan p;
  moe_status s = make_plan(cfg, &p);
  if (s != MOE_OK) return s;
  *bytes = p.L.total_bytes;
  return MOE_OK;
}

moe_status moe_workspace_layout_of(const moe_config* cfg, moe_workspace_layout* layout) {
  if (!layout) return MOE_ERR_INVALID_ARG;
  Plan p;
  moe_status s = make_plan(cfg, &p);
  if (s != MOE_OK) return s;
  *layout = p.L;
  return MOE_OK;
}

moe_status moe_workspace_init(const moe_config* cfg, void* ws, size_t ws_bytes, void* stream) {
  Plan p;
  moe_status s = make_plan(cfg, &p);
  if (s != MOE_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != MOE_OK) return s;
  cudaGetLastError();
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws_at<uint8_t>(ws, p.L.status), 0, 32, st) != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(cudaMemsetAsync(ws_at<uint8_t>(ws, p.stat_acc), 0, stats_acc_bytes(p.E), st));
}

moe_status moe_route(const moe_config* cfg, const void* x, const moe_weights* w, int32_t* idx, float* gate,
                     float* logits, float* probs, void* stats, void* ws, size_t ws_bytes, void* stream) {
  Plan p;
  moe_status s = make_plan(cfg, &p);
  if (s != MOE_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != MOE_OK) return s;
  if ((s = check_weights(p, w, true, false)) != MOE_OK) return s;
  if (!ok_opt(logits) || !ok_opt(probs) || !ok_opt(stats)) return MOE_ERR_INVALID_ARG;
  if (p.N == 0) return MOE_OK;
  if (!ok_ptr(x) || !ok_ptr(idx) || !ok_ptr(gate)) return MOE_ERR_INVALID_ARG;
  cudaGetLastError();
  if (p.sharded) {
    // one shard of a batch: the statistic partial sums stay in the workspace
    // (stat_acc) for the exchange; moe_permute_shard finalises them
    return cuda_status(launch_router(p, x, w, idx, gate, logits, probs, nullptr, ws, (cudaStream_t)stream,
                                     nullptr, false));
  }
  return do_route(p, x, w, idx, gate, logits, probs, stats, ws, (cudaStream_t)stream);
}

moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* idx, const float* gate, void* xp,
                       int32_t* tok_rows, int32_t* tok_off, int32_t* expert_off, int32_t* row_token,
                       float* row_gate, void* stats, void* ws, size_t ws_bytes, void* stream) {
  Plan p;
  moe_status s = make_plan(cfg, &p);
  if (s != MOE_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != MOE_OK) return s;
  if (!ok_opt(stats) || !ok_ptr(expert_off)) return MOE_ERR_INVALID_ARG;
  if (p.ec && !ok_ptr(tok_off)) return MOE_ERR_INVALID_ARG;
  if (p.sharded) return MOE_ERR_INVALID_ARG;  // a shard needs the other shards' counts: moe_permute_shard
  if (p.N == 0) {
    cudaGetLastError();
    return cuda_status(cudaMemsetAsync(expert_off, 0, (size_t)(p.E + 1) * 4, (cudaStream_t)stream));
  }
  if (!ok_ptr(x) || !ok_ptr(idx) || !ok_ptr(gate) || !ok_ptr(xp) || !ok_ptr(tok_rows) || !ok_ptr(row_token) ||
      !ok_ptr(row_gate))
    return MOE_ERR_INVALID_ARG;
  cudaGetLastError();
  return cuda_status(launch_permute(p, x, idx, gate, xp, tok_rows, tok_off, expert_off, row_token, row_gate, stats,
                                    ws, (cudaStream_t)stream, kCountsFromIdx));
}

moe_status moe_permute_shard(const moe_config* cfg, const void* x, const int32_t* idx, const float* gate,
                             const int32_t* shard_counts, int32_t n_shards, int32_t shard_rank, void* xp,
                             int32_t* tok_rows, int32_t* expert_off, int32_t* row_token, float* row_gate, void* stats,
                             void* ws, size_t ws_bytes, void* stream) {
  Plan p;
  moe_status s = make_plan(cfg, &p);
  if (s != MOE_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != MOE_OK) return s;
  if (p.ec) return MOE_ERR_UNSUPPORTED;
  if (n_shards < 1 || shard_rank < 0 || shard_rank >= n_shards) return MOE_ERR_INVALID_ARG;
  if (!ok_ptr(shard_counts) || !ok_opt(stats) || !ok_ptr(expert_off)) return MOE_ERR_INVALID_ARG;
  if (p.N > 0 && (!ok_ptr(x) || !ok_ptr(idx) || !ok_ptr(gate) || !ok_ptr(xp) || !ok_ptr(tok_rows) ||
                  !ok_ptr(row_token) || !ok_ptr(row_gate)))
    return MOE_ERR_INVALID_ARG;
  cudaGetLastError();
  cudaStream_t st = (cudaStream_t)stream;
  // the statistics are always finalised (into the workspace's copy when stats is NULL):
  // finalising also zeroes the partial sums for the next call
  void* st_buf = stats_or_ws(p, stats, ws);
  if (p.N == 0) {
    // an empty shard still finalises the exchanged statistics
    if (cudaMemsetAsync(expert_off, 0, (size_t)(p.E + 1) * 4, st) != cudaSuccess) return MOE_ERR_CUDA;
    return cuda_status(launch_router_stats_finalize(p, ws, st_buf, st));
  }
  return cuda_status(launch_permute(p, x, idx, gate, xp, tok_rows, nullptr, expert_off, row_token, row_gate, st_buf,
                                    ws, st, kCountsFromIdx, shard_counts, n_shards, shard_rank));
}

moe_status moe_expert_ffn(const moe_config* cfg, const void* xp, const int32_t* expert_off, const float* row_gate,
                          const void* x, const moe_weights* w, void* yp, void* ys, void* ws, size_t ws_bytes,
                          void* stream) {
  Plan p;
  moe_status s = make_plan(cfg, &p);
  if (s != MOE_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != MOE_OK) return s;
  if ((s = check_weights(p, w, false, true)) != MOE_OK) return s;
  if (p.N == 0) return MOE_OK;
  if (!ok_ptr(xp) || !ok_ptr(expert_off) || !ok_ptr(row_gate) || !ok_ptr(yp)) return MOE_ERR_INVALID_ARG;
  if (p.S > 0 && (!ok_ptr(x) || !ok_ptr(ys))) return MOE_ERR_INVALID_ARG;
  if (p.bf16 && !tc_gemm_available()) return MOE_ERR_CUDA;
  cudaGetLastError();
  return do_ffn(p, xp, expert_off, row_gate, x, w, yp, ys, ws, (cudaStream_t)stream, 3);
}

moe_status moe_combine(const moe_config* cfg, const void* yp, const int32_t* tok_rows, const int32_t* tok_off,
                       const void* ys, const void* x, void* out, void* stream) {
  Plan p;
  moe_status s = make_plan(cfg, &p);
  if (s != MOE_OK) return s;
  if (p.N == 0) return MOE_OK;
  if (!ok_ptr(yp) || !ok_ptr(tok_rows) || !ok_ptr(out) || !ok_opt(ys) || !ok_opt(x)) return MOE_ERR_INVALID_ARG;
  if (p.ec && !ok_ptr(tok_off)) return MOE_ERR_INVALID_ARG;
  if (p.passthrough && !x) return MOE_ERR_INVALID_ARG;
  cudaGetLastError();
  return cuda_status(launch_combine(p, yp, tok_rows, tok_off, ys, x, out, (cudaStream_t)stream));
}

namespace {

// Shared experts on a second stream (see moe_forward_overlap): their up- and
// down-projection launches, forked from `st` and joined back before the combine.
struct SideStream {
  cudaStream_t st;
  cudaEvent_t fork, join;
  int64_t ctas;
};

moe_status forward_impl(const Plan& p, const void* x, const moe_weights* w, void* out, void* stats, void* ws,
                        cudaStream_t st, void* const* events, int32_t n_events, const SideStream* side) {
  int ev = 0;
  auto mark = [&]() -> bool {
    if (ev < n_events && ev < 6) {
      if (cudaEventRecord((cudaEvent_t)events[ev], st) != cudaSuccess) return false;
    }
    ++ev;
    return true;
  };
  const moe_workspace_layout& L = p.L;
  int32_t* idx = ws_at<int32_t>(ws, L.idx);
  float* gate = ws_at<float>(ws, L.gate);
  int32_t* tok_rows = ws_at<int32_t>(ws, L.tok_rows);
  int32_t* tok_off = ws_at<int32_t>(ws, L.tok_off);
  int32_t* expert_off = ws_at<int32_t>(ws, L.expert_off);
  int32_t* row_token = ws_at<int32_t>(ws, L.row_token);
  float* row_gate = ws_at<float>(ws, L.row_gate);
  // MOE_FLAG_GATHER_ROWS: the up-projection gathers its rows from x by row_token (no xp copy)
  void* xp = p.gather ? nullptr : ws_at<uint8_t>(ws, L.xp);
  const int32_t* gather_rows = p.gather ? row_token : nullptr;
  void* yp = ws_at<uint8_t>(ws, L.yp);
  void* ys = p.S > 0 ? ws_at<uint8_t>(ws, L.ys) : nullptr;
  void* st_buf = stats_or_ws(p, stats, ws);
  moe_status s;
  // the main stream's GEMM launches: every family, or the routed experts only when the
  // shared experts run on the side stream
  const int fams = side ? kRoutedFamily : (kRoutedFamily | kSharedFamily);
  if (side) {
    void* h = ws_at<uint8_t>(ws, p.L.h);
    void* hs = ws_at<uint8_t>(ws, p.L.hs);
    if (cudaEventRecord(side->fork, st) != cudaSuccess || cudaStreamWaitEvent(side->st, side->fork, 0) != cudaSuccess)
      return MOE_ERR_CUDA;
    for (int part = 1; part <= 2; ++part)
      if (launch_ffn_bf16(p, xp, expert_off, row_gate, x, w, h, hs, yp, ys, status_ptr(p, ws), side->st, part,
                          nullptr, kSharedFamily, side->ctas) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaEventRecord(side->join, side->st) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (!mark()) return MOE_ERR_CUDA;
  int32_t* fused_counts = p.ec ? nullptr : ws_at<int32_t>(ws, p.tile_counts);
  const bool fused_offsets = permute_fuses_offsets(p);
  if ((s = do_route(p, x, w, idx, gate, ws_at<float>(ws, L.logits), p.ec ? ws_at<float>(ws, L.probs) : nullptr,
                    st_buf, ws, st, fused_counts)) != MOE_OK)
    return s;
  if (!mark()) return MOE_ERR_CUDA;
  const PermuteMode mode = p.ec ? kCountsFromIdx : (fused_offsets ? kFusedOffsets : kCountsFromRouter);
  if (launch_permute(p, x, idx, gate, xp, tok_rows, tok_off, expert_off, row_token, row_gate, st_buf, ws, st,
                     mode) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (!mark()) return MOE_ERR_CUDA;
  if ((s = do_ffn(p, xp, expert_off, row_gate, x, w, yp, ys, ws, st, 1, gather_rows, fams)) != MOE_OK) return s;
  if (!mark()) return MOE_ERR_CUDA;
  if ((s = do_ffn(p, xp, expert_off, row_gate, x, w, yp, ys, ws, st, 2, gather_rows, fams)) != MOE_OK) return s;
  if (!mark()) return MOE_ERR_CUDA;
  if (side && cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_combine(p, yp, tok_rows, tok_off, ys, x, out, st, side == nullptr) != cudaSuccess) return MOE_ERR_CUDA;
  if (!mark()) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status forward_checks(const Plan& p, const void* x, const moe_weights* w, void* out, void* stats, void* ws,
                          size_t ws_bytes) {
  moe_status s;
  if (p.sharded) return MOE_ERR_INVALID_ARG;  // a shard exchanges counts between route and permute
  if ((s = check_ws(p, ws, ws_bytes)) != MOE_OK) return s;
  if ((s = check_weights(p, w, true, true)) != MOE_OK) return s;
  if (!ok_opt(stats)) return MOE_ERR_INVALID_ARG;
  if (p.N == 0) return MOE_OK;
  if (!ok_ptr(x) || !ok_ptr(out)) return MOE_ERR_INVALID_ARG;
  if (p.bf16 && !tc_gemm_available()) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

moe_status moe_forward_traced(const moe_config* cfg, const void* x, const moe_weights* w, void* out, void* stats,
                              void* ws, size_t ws_bytes, void* stream, void* const* events, int32_t n_events) {
  Plan p;
  moe_status s = make_plan(cfg, &p);
  if (s != MOE_OK) return s;
  if ((s = forward_checks(p, x, w, out, stats, ws, ws_bytes)) != MOE_OK) return s;
  if (n_events > 0 && !events) return MOE_ERR_INVALID_ARG;
  if (p.N == 0) return MOE_OK;
  cudaGetLastError();
  return forward_impl(p, x, w, out, stats, ws, (cudaStream_t)stream, events, n_events, nullptr);
}

moe_status moe_forward(const moe_config* cfg, const void* x, const moe_weights* w, void* out, void* stats, void* ws,
                       size_t ws_bytes, void* stream) {
  return moe_forward_traced(cfg, x, w, out, stats, ws, ws_bytes, stream, nullptr, 0);
}

moe_status moe_forward_overlap(const moe_config* cfg, const void* x, const moe_weights* w, void* out, void* stats,
                               void* ws, size_t ws_bytes, void* stream, void* side_stream, void* ev_fork,
                               void* ev_join, int32_t side_ctas) {
  Plan p;
  moe_status s = make_plan(cfg, &p);
  if (s != MOE_OK) return s;
  if ((s = forward_checks(p, x, w, out, stats, ws, ws_bytes)) != MOE_OK) return s;
  if (!side_stream || side_stream == stream || !ev_fork || !ev_join || side_ctas < 0) return MOE_ERR_INVALID_ARG;
  if (p.N == 0) return MOE_OK;
  cudaGetLastError();
  if (!p.bf16 || p.S == 0)  // nothing to overlap (fp32 layers run their shared experts in line)
    return forward_impl(p, x, w, out, stats, ws, (cudaStream_t)stream, nullptr, 0, nullptr);
  SideStream side{(cudaStream_t)side_stream, (cudaEvent_t)ev_fork, (cudaEvent_t)ev_join, side_ctas};
  return forward_impl(p, x, w, out, stats, ws, (cudaStream_t)stream, nullptr, 0, &side);
}

moe_status moe_get_device_status(const moe_config* cfg, void* ws, size_t ws_bytes, void* stream,
                                 int32_t* device_error) {
  Plan p;
  moe_status s = make_plan(cfg, &p);
  if (s != MOE_OK) return s;
  if ((s = check_ws(p, ws, ws_bytes)) != MOE_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  int32_t word[4] = {0, 0, 0, 0};
  cudaGetLastError();
  if (cudaMemcpyAsync(word, ws_at<uint8_t>(ws, p.L.status), sizeof word, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(ws_at<uint8_t>(ws, p.L.status), 0, sizeof word, st) != cudaSuccess) return MOE_ERR_CUDA;
  // (the ticket after the error word is left alone: it is zero between calls)
  if (device_error) *device_error = word[0];
  if (word[0] & kErrTimeout) return MOE_ERR_TIMEOUT;
  if (word[0] & kErrIndex) return MOE_ERR_DEVICE_CHECK;
  return MOE_OK;
}

}  // extern "C"
