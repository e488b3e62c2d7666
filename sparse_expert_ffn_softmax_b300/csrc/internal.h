// Internal launch interface of the library (host side). Not installed.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kRouterWarps = 8;
constexpr int kMaxTileTokens = 32;  // a tile is ranked by one warp, one token per lane

// Everything the launchers need, derived once from a validated moe_config.
struct Plan {
  moe_config cfg;
  int64_t N, d, F, E, S, Fs, k;
  int64_t Ntot;       // tokens of the whole batch (N unless the batch is sharded over calls)
  bool sharded;       // Ntot > N: this call holds one contiguous token shard of the batch
  bool passthrough;   // MOE_FLAG_DROP_PASSTHROUGH
  bool gather;        // MOE_FLAG_GATHER_ROWS (bf16): the up-projection gathers its rows from x
  bool fp8w;          // MOE_WEIGHTS_MXFP8: routed expert weights are E4M3 codes with E8M0 block scales
  bool bf16, swiglu, ec, bias;
  int64_t cap;       // C
  int64_t max_rows;  // rows reserved for xp / h / yp
  int64_t tile;      // tokens per tile (8, 16 or 32): one router block, one permute block
  int64_t tiles;     // ceil(N / tile)
  int64_t words;     // ceil(E / 32): expert bitmap words per token (expert choice)
  moe_workspace_layout L;
  // scratch sub-buffers (byte offsets into the workspace)
  size_t stat_acc;                    // fixed-point router statistic accumulators (stats.cuh)
  size_t tile_counts, tile_base;      // permute [E][T], [E][T+1]
  size_t ec_bits;                     // [N][words]
  size_t probs_t;                     // fp32 [E][N] (expert choice): each expert's probabilities in token order
  int64_t rsplit;                     // bf16 router GEMM split along K into this many groups (1: none)
  size_t logits_part;                 // [rsplit][N][E] fp32 partial logits when rsplit > 1
  size_t rank_base;                   // int32 [E]: assignments to each expert in earlier shards
};

// K groups of the bf16 logits GEMM (layers with more than 32 experts) for a batch
// of N tokens, a function of the shapes alone: fewer than 75 128-token tiles leave at
// least half the SMs idle, so the K range is split into floor(148 / tiles) equal
// groups (each keeping >= 4 K blocks), whose partial sums the routing kernel adds in
// order (measured on the 8192-token, 160-expert layer: route 69.8 -> 66.7 us with two).
constexpr int64_t kRouterTcMinE = 33;        // bf16 layers with more experts route from tensor-core logits
constexpr int64_t kRouterSplitMaxTiles = 75;  // K split only below this many 128-token tiles
int64_t router_k_splits(int64_t N, int64_t d, int64_t E);

moe_status make_plan(const moe_config* cfg, Plan* p);

inline int32_t* status_ptr(const Plan& p, void* ws) {
  return reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + p.L.status);
}
template <typename T>
inline T* ws_at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// router.cu. One router block per 32-token tile. tile_counts (nullable) receives
// the per-tile expert counts [E][T] for the permute. finalize: reduce the
// statistics in a separate kernel (stand-alone routing and expert choice);
// otherwise a later kernel of the forward reduces the router's partials.
cudaError_t launch_router(const Plan& p, const void* x, const moe_weights* w, int32_t* idx, float* gate,
                          float* logits, float* probs, void* stats, void* ws, cudaStream_t st,
                          int32_t* tile_counts, bool finalize);
// Router statistics from the workspace's accumulators (which it then zeroes).
cudaError_t launch_router_stats_finalize(const Plan& p, void* ws, void* stats, cudaStream_t st);
// True when the router writes the logits to memory before a second kernel reads
// them (bf16 layers that the fused tensor-core router does not cover).
bool router_uses_tc(const Plan& p);

// permute.cu. Token choice needs per-tile expert counts and their prefix:
//  kCountsFromIdx    count them from idx (stand-alone moe_permute);
//  kCountsFromRouter the router wrote the counts; the scan kernel also
//                    finalises the router statistics;
//  kFusedOffsets     the router wrote the counts and every scatter block derives
//                    its prefixes and the expert offsets itself (small E x T,
//                    permute_fuses_offsets); scatter block 0 finalises the statistics.
enum PermuteMode { kCountsFromIdx = 0, kCountsFromRouter = 1, kFusedOffsets = 2 };
bool permute_fuses_offsets(const Plan& p);
// probs_t (nullable): room for an expert-major copy of the probabilities [E][N], read
// by the selection instead of the strided columns of probs.
cudaError_t launch_ec_select(const Plan& p, const float* probs, int32_t* idx, float* gate, float* probs_t,
                             cudaStream_t st);
// xp null: only the row metadata is written (the up-projection gathers the rows from x).
// shard_counts (token-sharded batch, kCountsFromIdx only): [n_shards][E] assignment
// counts of every shard before dropping; the ranks of this shard's assignments start
// after those of shards 0 .. shard_rank - 1.
cudaError_t launch_permute(const Plan& p, const void* x, const int32_t* idx, const float* gate, void* xp,
                           int32_t* tok_rows, int32_t* tok_off, int32_t* expert_off, int32_t* row_token,
                           float* row_gate, void* stats, void* ws, cudaStream_t st, PermuteMode mode,
                           const int32_t* shard_counts = nullptr, int32_t n_shards = 0, int32_t shard_rank = 0);
// x: the layer input, read for tokens with no kept row when p.passthrough (else unused).
// pdl false: an ordinary launch (after a cross-stream event wait).
cudaError_t launch_combine(const Plan& p, const void* yp, const int32_t* tok_rows, const int32_t* tok_off,
                           const void* ys, const void* x, void* out, cudaStream_t st, bool pdl = true);

// ffn_simt.cu (fp32 layers)
cudaError_t launch_ffn_f32(const Plan& p, const void* xp, const int32_t* expert_off, const float* row_gate,
                           const void* x, const moe_weights* w, void* h, void* hs, void* yp, void* ys,
                           int32_t* status, cudaStream_t st, int part);

// gemm_tc.cu (bf16 layers, tcgen05)
// gather_rows non-null: the routed up-projection gathers its rows from x by these row
// ids (tile::gather4) instead of reading xp. families: kRoutedFamily | kSharedFamily
// (the routed experts' and the shared experts' tiles of each launch); grid_cap > 0
// limits the CTAs of each launch (the rest of the SMs stay free for other streams).
constexpr int kRoutedFamily = 1, kSharedFamily = 2;
cudaError_t launch_ffn_bf16(const Plan& p, const void* xp, const int32_t* expert_off, const float* row_gate,
                            const void* x, const moe_weights* w, void* h, void* hs, void* yp, void* ys,
                            int32_t* status, cudaStream_t st, int part, const int32_t* gather_rows = nullptr,
                            int families = kRoutedFamily | kSharedFamily, int64_t grid_cap = 0);
bool tc_gemm_available();
// Router logits x W_r^T on the tensor cores (bf16 layers), fp32: splits = 1 writes
// logits + logit_bias [N, E]; splits > 1 writes [splits][N][E] partial sums over
// equal K ranges without the bias (splits divides d / 64).
cudaError_t launch_router_logits_tc(const Plan& p, const void* x, const void* w_router, const float* logit_bias,
                                    float* out, int splits, int32_t* status, cudaStream_t st);

}  // namespace moe
