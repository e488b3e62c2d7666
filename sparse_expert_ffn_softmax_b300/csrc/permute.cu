// Capacity, in-token-order dropping, permutation into expert-contiguous rows,
// expert-choice selection, and the combine back into token order.
//
// Pages: "Mixture of Experts" (aigrafen.se) "Expert capacity" (C = tokens /
// experts x capacity factor; tokens above the limit are dropped) and its MoE
// code (each expert's tokens listed in index order and cut to the first C);
// "MoE Architecture" (vanos001.github.io) CapacityManagedMoE and
// ExpertChoiceRouter; "Mixture of Experts (MoE)" (wiki.ai-engineering.at)
// "Gather/scatter outputs from experts".
//
// Token choice runs four kernels, none of which waits on another block:
//  1. count:   one warp per tile of 32 consecutive tokens counts the tile's
//              assignments per expert            -> tile_counts[E][T]
//  2. scan:    one warp per expert, exclusive prefix over tiles
//                                                -> tile_base[E][T+1] (last = total)
//  3. offsets: one block; kept_e = min(count_e, C), expert_off = exclusive
//              prefix of kept, dropped / rows statistics
//  4. scatter: one warp per tile; the in-tile rank of (t, j) among the tile's
//              tokens that chose the same expert comes from a per-warp bitmask
//              of lanes per expert (atomicOr, then popc of the lower lanes), so
//              rank = tile_base + in-tile rank is the token-order rank exactly.
//              Kept pairs get row = expert_off[e] + rank; the warp then copies
//              each of its tokens' rows of x into xp with 16-byte vectors (x is
//              read once, written once per kept choice).
// Expert choice: one block per expert radix-selects the C-th largest
// probability (4 passes of 8 bits over the column), takes every larger one and
// the first ties in token order, and lists them in ascending token order; a
// bitmap of (token, expert) then gives each token its rows in ascending expert
// order (a CSR: tok_off / tok_rows) for the copy and the combine.
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "mx.cuh"
#include "offsets.cuh"
#include "stats.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32) count_kernel(const int32_t* __restrict__ idx, int64_t N, int64_t k,
                                                            int64_t E, int64_t T, int64_t TT,
                                                            int32_t* __restrict__ tile_counts, int32_t* status) {
  extern __shared__ int32_t s_hist[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t tile = (int64_t)blockIdx.x * kWarps + warp;
  if (tile >= T) return;
  int32_t* h = s_hist + warp * E;
  for (int64_t e = lane; e < E; e += 32) h[e] = 0;
  __syncwarp();
  const int64_t t = tile * TT + lane;
  if (lane < TT && t < N) {
    for (int64_t j = 0; j < k; ++j) {
      const int32_t e = idx[t * k + j];
      if (e < 0 || e >= E) {
        record_error(status, kErrIndex, 101, (int32_t)t, e);
        continue;
      }
      atomicAdd(&h[e], 1);
    }
  }
  __syncwarp();
  for (int64_t e = lane; e < E; e += 32) tile_counts[e * T + tile] = h[e];
}

struct RouterStatsArgs {  // finalise the router statistics from these accumulators (acc.p null: no)
  StatsAcc acc;
  float alpha;
};

// Phase 1 (every block): one warp per expert, exclusive prefix of its tile
// counts over the tiles -> tile_base[e][0..T-1], total in tile_base[e][T].
// Phase 2 (the last block to finish, found with an atomic ticket; no block waits
// for another): kept_e = min(count_e, C), expert_off = exclusive prefix of kept,
// the dropping statistics and, when given the router partials, the router
// statistics.
// n_stats: tokens the router statistics average over (the whole batch when sharded);
// rank_base: per-expert assignments in earlier shards, or null.
__global__ void __launch_bounds__(kWarps * 32) scan_offsets_kernel(
    const int32_t* __restrict__ tile_counts, int64_t E, int64_t T, int64_t cap, int64_t N, int64_t k,
    int32_t* __restrict__ tile_base, int32_t* __restrict__ expert_off, void* stats, int32_t* ticket,
    RouterStatsArgs rs, int64_t n_stats, const int32_t* __restrict__ rank_base) {
  const int warp = threadIdx.x >> 5;
  const int64_t e = (int64_t)blockIdx.x * kWarps + warp;
  if (e < E) scan_expert_tiles(tile_counts + e * T, tile_base + e * (T + 1), T);
  if (!last_block_ticket(ticket)) return;
  offsets_from_totals(tile_base, E, T, cap, N, k, expert_off, stats, rank_base);
  if (stats && rs.acc.p) finalize_router_stats(rs.acc, n_stats, E, k, cap, 0, rs.alpha, stats);
}

// Token-sharded batch: base[e] = assignments to expert e in shards 0 .. rank - 1,
// from every shard's counts [n_shards][E] (the ranks of this shard's assignments
// to e start there, in token order across the whole batch).
__global__ void shard_base_kernel(const int32_t* __restrict__ shard_counts, int32_t n_shards, int32_t rank,
                                  int64_t E, int32_t* __restrict__ base, int32_t* status) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  int64_t b = 0;
  for (int32_t r = 0; r < rank && r < n_shards; ++r) b += shard_counts[(int64_t)r * E + e];
  if (b < 0 || b > 0x7fffffff) {
    record_error(status, kErrIndex, 105, (int32_t)e, rank);
    b = 0;
  }
  base[e] = (int32_t)b;
}

// One block per tile of 8-32 tokens. Warp 0 ranks the tile's (token, choice)
// pairs: the in-tile rank among the tile's tokens that chose the same expert is
// the popcount of the lower lanes in a per-expert lane mask, so rank =
// (assignments to e in earlier tiles) + in-tile rank is the exact token-order
// rank. Kept pairs get row = expert_off[e] + rank. Then all 8 warps copy the
// tile's token rows of x into xp with 16-byte vectors (each x row read once,
// written once per kept choice).
// kFused: the block itself derives what it needs from the router's per-tile
// counts [E][T] -- the count of each expert in earlier tiles, the totals, and
// expert_off (every block computes the same integers; block 0 also writes
// expert_off and the dropping statistics) -- so no scan kernel runs before it;
// one extra block (blockIdx.x == T) turns the router's accumulators into the
// router statistics.
// Otherwise tile_base [E][T+1] and expert_off come from scan_offsets_kernel.
// rank_base (token-sharded batch, else null): assignments to each expert in earlier
// shards; (t, j) is kept when rank_base[e] + its rank in this shard < C.
// MXFP8 rows (bf16 layers whose routed experts compute in MXFP8): a lane's 16-byte
// chunk is 8 values of the row and lanes 4q .. 4q + 3 hold one 32-value MX block (the
// chunks a warp covers start at a multiple of 4). Returns the lane's 8 E4M3 codes and,
// in sb, the block's E8M0 scale byte. Every lane of the warp takes part.
__device__ __forceinline__ uint2 mx_chunk(uint4 v, uint32_t& sb) {
  float f[8];
  Vec16<__nv_bfloat16>::unpack(v, f);
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
  amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
  sb = mx::scale_byte(amax);
  const float inv = mx::inv_scale(sb);
  return make_uint2(mx::e4m3x4(f[0] * inv, f[1] * inv, f[2] * inv, f[3] * inv),
                    mx::e4m3x4(f[4] * inv, f[5] * inv, f[6] * inv, f[7] * inv));
}

template <typename DT, bool kFused>
__global__ void __launch_bounds__(kWarps * 32) scatter_kernel(
    const DT* __restrict__ x, const int32_t* __restrict__ idx, const float* __restrict__ gate,
    const int32_t* __restrict__ counts_or_base, int32_t* __restrict__ expert_off, int64_t N, int64_t d, int64_t k,
    int64_t E, int64_t T, int64_t TT, int64_t cap, DT* __restrict__ xp, int32_t* __restrict__ tok_rows,
    int32_t* __restrict__ row_token, float* __restrict__ row_gate, void* stats, int32_t* status,
    RouterStatsArgs rs, const int32_t* __restrict__ rank_base, uint8_t* __restrict__ xs) {
  // blockIdx.y selects a slice of the row's 16-byte chunks: small batches copy
  // their rows with more blocks. Every slice ranks the tile (cheap); slice 0
  // writes the row metadata. xs non-null (bf16, MXFP8 experts): xp receives the rows'
  // E4M3 codes [rows, d] and xs their E8M0 scales [rows, d / 32].
  const bool meta = blockIdx.y == 0;
  extern __shared__ uint32_t s_dyn[];
  pdl_wait();
  pdl_launch_next();
  uint32_t* msk = s_dyn;                                       // [E]
  int32_t* s_rows = reinterpret_cast<int32_t*>(s_dyn + E);     // [32][k]
  int32_t* s_pre = s_rows + kMaxTileTokens * k;                // [E]   (kFused)
  int32_t* s_off = s_pre + E;                                  // [E+1] (kFused)
  __shared__ int s_warp[33];
  using VT = Vec16<DT>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t tile = blockIdx.x;
  if (tile >= T) {  // the extra block: router statistics, off the other blocks' path
    if (stats && rs.acc.p && blockIdx.y == 0) finalize_router_stats(rs.acc, N, E, k, cap, 0, rs.alpha, stats);
    return;
  }
  if (kFused) {
    // each expert's counts in earlier tiles and in all tiles (E * T <= 8192): few tiles
    // (decode batches), one thread per expert along its T counts, loads in flight
    // together; many tiles, one warp per expert with its lanes striding over them
    if (T <= 64) {
      for (int64_t e = threadIdx.x; e < E; e += blockDim.x) {
        const int32_t* cnt = counts_or_base + e * T;
        int pre = 0, tot = 0;
#pragma unroll 8
        for (int64_t t = 0; t < T; ++t) {
          const int c = cnt[t];
          tot += c;
          pre += t < tile ? c : 0;
        }
        s_pre[e] = pre;
        s_off[e] = tot;  // totals for now, offsets below
      }
    } else {
      for (int64_t e = warp; e < E; e += kWarps) {
        const int32_t* cnt = counts_or_base + e * T;
        int pre = 0, tot = 0;
#pragma unroll 4
        for (int64_t t = lane; t < T; t += 32) {
          const int c = cnt[t];
          tot += c;
          pre += t < tile ? c : 0;
        }
        pre = warp_sum_int(pre);
        tot = warp_sum_int(tot);
        if (lane == 0) {
          s_pre[e] = pre;
          s_off[e] = tot;
        }
      }
    }
    __syncthreads();
    const int per = (int)ceil_div(E, (int64_t)blockDim.x);  // <= 2
    const int64_t e0 = (int64_t)threadIdx.x * per;
    int kept[2] = {0, 0}, ksum = 0, dsum = 0;
    for (int i = 0; i < per && i < 2; ++i)
      if (e0 + i < E) {
        const int tot = s_off[e0 + i];
        const int64_t cl = cap_left(cap, rank_base, e0 + i);
        kept[i] = (int)(tot < cl ? tot : cl);
        ksum += kept[i];
        dsum += tot - kept[i];
      }
    int rows = 0, dropped = 0;
    const bool first = blockIdx.x == 0 && blockIdx.y == 0;
    int off = block_exclusive_scan(ksum, s_warp, &rows);  // (syncs: all totals read before overwritten)
    if (first) block_exclusive_scan(dsum, s_warp, &dropped);
    for (int i = 0; i < per && i < 2; ++i)
      if (e0 + i < E) {
        s_off[e0 + i] = off;
        if (first) expert_off[e0 + i] = off;
        off += kept[i];
      }
    if (threadIdx.x == 0) {
      s_off[E] = rows;
      if (first) expert_off[E] = rows;
    }
    if (first && stats) {
      moe_stats_header* hdr = static_cast<moe_stats_header*>(stats);
      int32_t* kept_out = reinterpret_cast<int32_t*>(reinterpret_cast<float*>(hdr + 1) + 2 * E) + E;
      for (int i = 0; i < per && i < 2; ++i)
        if (e0 + i < E) kept_out[e0 + i] = kept[i];
      if (threadIdx.x == 0) {
        hdr->dropped = dropped;
        hdr->dropped_share = (float)((double)dropped / (double)(N * k));
        hdr->capacity = (int32_t)cap;
        hdr->rows = rows;
        hdr->n_experts = (int32_t)E;
      }
    }
    __syncthreads();
  }
  if (warp == 0) {
    const int64_t t = tile * TT + lane;
    const bool valid = lane < TT && t < N;
    const uint32_t lt = (1u << lane) - 1u;
    if (valid)
      for (int64_t j = 0; j < k; ++j) {
        const int32_t e = idx[t * k + j];
        if (e >= 0 && e < E) msk[e] = 0u;
      }
    __syncwarp();
    if (valid)
      for (int64_t j = 0; j < k; ++j) {
        const int32_t e = idx[t * k + j];
        if (e >= 0 && e < E) {
          const uint32_t old = atomicOr(&msk[e], 1u << lane);
          if ((old & (1u << lane)) && meta) record_error(status, kErrIndex, 104, (int32_t)t, e);  // listed twice
        }
      }
    __syncwarp();
    for (int64_t j = 0; j < k; ++j) {
      int32_t row = -1;
      if (valid) {
        const int32_t e = idx[t * k + j];
        if (e >= 0 && e < E) {
          const int64_t before = kFused ? s_pre[e] : counts_or_base[(int64_t)e * (T + 1) + tile];
          const int64_t r = before + __popc(msk[e] & lt);  // rank among this shard's assignments to e
          if (r < cap_left(cap, rank_base, e)) {
            row = (kFused ? s_off[e] : expert_off[e]) + (int32_t)r;
            if (meta) {
              row_token[row] = (int32_t)t;
              row_gate[row] = gate[t * k + j];
            }
          }
        } else if (meta) {
          record_error(status, kErrIndex, 102, (int32_t)t, e);
        }
        if (meta) tok_rows[t * k + j] = row;
      }
      s_rows[lane * k + j] = row;
    }
  }
  __syncthreads();
  if (xp == nullptr) return;  // metadata only: the up-projection gathers the rows from x
  const int64_t nchunk = d / VT::n;
  int64_t cs = ceil_div(nchunk, (int64_t)gridDim.y);
  if (xs) cs = (cs + 3) & ~(int64_t)3;  // slices of whole MX blocks
  const int64_t cbeg = (int64_t)blockIdx.y * cs, cend = cbeg + cs < nchunk ? cbeg + cs : nchunk;
  if constexpr (std::is_same<DT, __nv_bfloat16>::value) {
    if (xs) {
      uint8_t* xq = reinterpret_cast<uint8_t*>(xp);
      for (int tt = warp; tt < TT; tt += kWarps) {
        const int64_t tok = tile * TT + tt;
        if (tok >= N) break;
        const int32_t my_row = lane < k ? s_rows[tt * k + lane] : -1;
        const uint4* src = reinterpret_cast<const uint4*>(x) + tok * nchunk;
        for (int64_t c0 = cbeg; c0 < cend; c0 += 32) {
          const int64_t c = c0 + lane;
          const bool act = c < cend;
          const uint4 v = act ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
          uint32_t sb;
          const uint2 q = mx_chunk(v, sb);
          for (int j = 0; j < k; ++j) {
            const int32_t row = __shfl_sync(kFull, my_row, j);
            if (act && row >= 0) {
              *reinterpret_cast<uint2*>(xq + (int64_t)row * d + c * 8) = q;
              if ((c & 3) == 0) xs[(int64_t)row * (d / 32) + (c >> 2)] = (uint8_t)sb;
            }
          }
        }
      }
      return;
    }
  }
  // each lane keeps kCopyUnroll 16-byte loads of the row in flight before the stores
  constexpr int kCopyUnroll = 4;
  for (int tt = warp; tt < TT; tt += kWarps) {
    const int64_t tok = tile * TT + tt;
    if (tok >= N) break;
    const int32_t my_row = lane < k ? s_rows[tt * k + lane] : -1;
    const uint4* src = reinterpret_cast<const uint4*>(x) + tok * nchunk;
    for (int64_t c0 = cbeg; c0 < cend; c0 += 32 * kCopyUnroll) {
      uint4 v[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t c = c0 + 32 * u + lane;
        v[u] = c < cend ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
      }
      for (int j = 0; j < k; ++j) {
        const int32_t row = __shfl_sync(kFull, my_row, j);  // the same in every lane
        if (row < 0) continue;
        uint4* dst = reinterpret_cast<uint4*>(xp) + (int64_t)row * nchunk;
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
          const int64_t c = c0 + 32 * u + lane;
          if (c < cend) dst[c] = v[u];
        }
      }
    }
  }
}

// ---- expert choice -----------------------------------------------------------

// probs [N, E] -> probs_t [E, N] through 32 x 32 tiles in shared memory (both sides coalesced).
__global__ void __launch_bounds__(32 * 8) ec_transpose_kernel(const float* __restrict__ probs, int64_t N, int64_t E,
                                                              float* __restrict__ probs_t) {
  __shared__ float tile[32][33];
  const int64_t t0 = (int64_t)blockIdx.x * 32, e0 = (int64_t)blockIdx.y * 32;
  const int lx = threadIdx.x & 31, ly = threadIdx.x >> 5;
  for (int r = ly; r < 32; r += 8) {
    const int64_t t = t0 + r, e = e0 + lx;
    tile[r][lx] = t < N && e < E ? probs[t * E + e] : 0.f;
  }
  __syncthreads();
  for (int r = ly; r < 32; r += 8) {
    const int64_t e = e0 + r, t = t0 + lx;
    if (e < E && t < N) probs_t[e * N + t] = tile[lx][r];
  }
}

// One block per expert over its probabilities, p(e, t) = probs[e * se + t * st] (se = N,
// st = 1 for the expert-major copy; se = 1, st = E for [N, E]): the C-th largest by four
// radix passes of 8 bits, then every larger one and the first ties in token order.
__global__ void __launch_bounds__(1024) ec_select_kernel(const float* __restrict__ probs, int64_t se, int64_t st,
                                                         int64_t N, int64_t E, int64_t cap,
                                                         int32_t* __restrict__ idx, float* __restrict__ gate) {
  __shared__ int hist[256];
  __shared__ int s_warp[33];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  const int64_t e = blockIdx.x;
  uint32_t prefix = 0, pmask = 0;
  if (threadIdx.x == 0) s_remaining = (int)cap;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    // (N rounded up to whole blocks so every lane of a warp takes part in the match;
    // probabilities crowd into a few bins, so lanes with equal bins add once together)
    const int64_t n_up = (N + blockDim.x - 1) / blockDim.x * blockDim.x;
    for (int64_t t = threadIdx.x; t < n_up; t += blockDim.x) {
      const uint32_t u = t < N ? __float_as_uint(probs[e * se + t * st]) : 0u;  // p >= 0: bit order = value order
      const bool in = t < N && (u & pmask) == prefix;
      const uint32_t bin = in ? (u >> shift) & 255u : 256u;
      const uint32_t same = __match_any_sync(kFull, bin);
      if (in && (__ffs(same) - 1) == (int)(threadIdx.x & 31)) atomicAdd(&hist[bin], __popc(same));
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int acc = 0, rem = s_remaining, b = 255;
      for (; b > 0; --b) {
        if (acc + hist[b] >= rem) break;
        acc += hist[b];
      }
      s_remaining = rem - acc;
      s_prefix = prefix | ((uint32_t)b << shift);
    }
    __syncthreads();
    prefix = s_prefix;
    pmask |= 255u << shift;
  }
  const uint32_t thr = prefix;
  const int need = s_remaining;  // ties equal to thr to take, first in token order
  int carry_eq = 0, carry_sel = 0;
  for (int64_t base = 0; base < N; base += blockDim.x) {
    const int64_t t = base + threadIdx.x;
    const uint32_t u = t < N ? __float_as_uint(probs[e * se + t * st]) : 0u;
    const int gt = (t < N && u > thr) ? 1 : 0;
    const int eq = (t < N && u == thr) ? 1 : 0;
    int tot_eq = 0, tot_sel = 0;
    const int eq_rank = block_exclusive_scan(eq, s_warp, &tot_eq) + carry_eq;
    const int sel = gt | (eq & (eq_rank < need ? 1 : 0));
    const int pos = block_exclusive_scan(sel, s_warp, &tot_sel) + carry_sel;
    if (sel && pos < cap) {
      idx[e * cap + pos] = (int32_t)t;
      gate[e * cap + pos] = __uint_as_float(u);
    }
    carry_eq += tot_eq;
    carry_sel += tot_sel;
  }
}

__global__ void ec_mark_kernel(const int32_t* __restrict__ idx, const float* __restrict__ gate, int64_t N,
                               int64_t E, int64_t cap, int64_t words, uint32_t* __restrict__ bits,
                               int32_t* __restrict__ row_token, float* __restrict__ row_gate,
                               int32_t* __restrict__ expert_off, int32_t* __restrict__ tok_off, int32_t* status) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i <= E) expert_off[i] = (int32_t)(i * cap);
  if (i >= E * cap) return;
  const int64_t e = i / cap;
  const int32_t t = idx[i];
  row_gate[i] = gate[i];
  row_token[i] = t;
  if (t < 0 || t >= N) {
    record_error(status, kErrIndex, 103, (int32_t)i, t);
    return;
  }
  atomicOr(&bits[(int64_t)t * words + (e >> 5)], 1u << (e & 31));
  atomicAdd(&tok_off[t], 1);  // the token's row count (zeroed before), scanned next
}

// tok_off[t] holds token t's row count (ec_mark_kernel); each thread turns a contiguous
// run of them into exclusive offsets in place.
__global__ void __launch_bounds__(1024) ec_tok_scan_kernel(int64_t N, int64_t E, int64_t cap,
                                                           int32_t* __restrict__ tok_off, void* stats) {
  __shared__ int s_warp[33];
  const int64_t per = ceil_div(N, (int64_t)blockDim.x);
  const int64_t t0 = (int64_t)threadIdx.x * per;
  const int64_t t1 = t0 + per < N ? t0 + per : N;
  int local = 0;
  for (int64_t t = t0; t < t1; ++t) local += tok_off[t];
  int total = 0;
  int run = block_exclusive_scan(local, s_warp, &total);
  for (int64_t t = t0; t < t1; ++t) {
    const int c = tok_off[t];
    tok_off[t] = run;
    run += c;
  }
  if (threadIdx.x == 0) tok_off[N] = total;
  if (stats && threadIdx.x == 0) {
    moe_stats_header* hdr = static_cast<moe_stats_header*>(stats);
    hdr->dropped = 0;
    hdr->dropped_share = 0.f;
    hdr->capacity = (int32_t)cap;
    hdr->rows = (int32_t)(E * cap);
    hdr->n_experts = (int32_t)E;
  }
  if (stats) {
    moe_stats_header* hdr = static_cast<moe_stats_header*>(stats);
    int32_t* kept_out = reinterpret_cast<int32_t*>(reinterpret_cast<float*>(hdr + 1) + 2 * E) + E;
    for (int64_t e = threadIdx.x; e < E; e += blockDim.x) kept_out[e] = (int32_t)cap;
  }
}

// One warp per token: its experts in ascending id, each located in that
// expert's ascending token list by binary search -> rows e*C + c.
__global__ void __launch_bounds__(kWarps * 32) ec_fill_kernel(const uint32_t* __restrict__ bits,
                                                              const int32_t* __restrict__ idx,
                                                              const int32_t* __restrict__ tok_off, int64_t N,
                                                              int64_t words, int64_t cap,
                                                              int32_t* __restrict__ tok_rows) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (t >= N) return;
  const uint32_t word = lane < words ? bits[t * words + lane] : 0u;
  const int c = __popc(word);
  const int excl = warp_inclusive_scan(c) - c;
  int pos = tok_off[t] + excl;
  uint32_t wleft = word;
  while (wleft) {
    const int b = __ffs(wleft) - 1;
    wleft &= wleft - 1;
    const int64_t e = (int64_t)lane * 32 + b;
    const int32_t* list = idx + e * cap;
    int64_t lo = 0, hi = cap;  // first position with list[pos] >= t
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if (list[mid] < t) lo = mid + 1; else hi = mid;
    }
    tok_rows[pos++] = (int32_t)(e * cap + lo);
  }
}

// Copy x rows into xp by a token's row list (expert choice CSR).
template <typename T>
__global__ void __launch_bounds__(kWarps * 32) copy_rows_csr_kernel(const T* __restrict__ x,
                                                                    const int32_t* __restrict__ tok_rows,
                                                                    const int32_t* __restrict__ tok_off, int64_t N,
                                                                    int64_t d, T* __restrict__ xp,
                                                                    uint8_t* __restrict__ xs) {
  using VT = Vec16<T>;
  const int lane = threadIdx.x & 31;
  const int64_t nchunk = d / VT::n;
  for (int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); t < N; t += (int64_t)gridDim.x * kWarps) {
    const int32_t beg = tok_off[t], n = tok_off[t + 1] - beg;
    const uint4* src = reinterpret_cast<const uint4*>(x) + t * nchunk;
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
      if (xs) {  // MXFP8 rows: codes into xp, scales into xs (see scatter_kernel)
        uint8_t* xq = reinterpret_cast<uint8_t*>(xp);
        for (int64_t c0 = 0; c0 < nchunk; c0 += 32) {
          const int64_t c = c0 + lane;
          const bool act = c < nchunk;
          const uint4 v = act ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
          uint32_t sb;
          const uint2 q = mx_chunk(v, sb);
          for (int i = 0; act && i < n; ++i) {
            const int64_t row = tok_rows[beg + i];
            *reinterpret_cast<uint2*>(xq + row * d + c * 8) = q;
            if ((c & 3) == 0) xs[row * (d / 32) + (c >> 2)] = (uint8_t)sb;
          }
        }
        continue;
      }
    }
    for (int64_t c = lane; c < nchunk; c += 32) {
      const uint4 v = __ldg(src + c);
      for (int i = 0; i < n; ++i) reinterpret_cast<uint4*>(xp)[(int64_t)tok_rows[beg + i] * nchunk + c] = v;
    }
  }
}

// out[t] = ys[t] + sum of yp over t's rows in list order: fp32 inputs, fp32
// accumulation, one rounding to the output type. A lane owns 16 output bytes.
// The first KU rows of a token are loaded together (all loads in flight before
// the first add); rows past KU follow one at a time. Same order of additions.
// x non-null (dropped-token pass-through): a token with no kept row gets x[t]
// added after ys[t].
template <typename TO, int KU>
__global__ void __launch_bounds__(kWarps * 32) combine_kernel(const float* __restrict__ yp,
                                                              const int32_t* __restrict__ tok_rows,
                                                              const int32_t* __restrict__ tok_off,
                                                              const float* __restrict__ ys, int64_t N, int64_t d,
                                                              int64_t k, TO* __restrict__ out,
                                                              const TO* __restrict__ x) {
  pdl_wait();
  pdl_launch_next();
  using VO = Vec16<TO>;
  constexpr int VN = VO::n;  // outputs per lane chunk: 8 (bf16) or 4 (fp32)
  constexpr int NV = VN / 4; // float4 loads per row and chunk
  const int lane = threadIdx.x & 31;
  const int64_t nchunk = d / VN;
  // blockIdx.y selects a slice of the row's chunks (more blocks for small batches)
  const int64_t cs = ceil_div(nchunk, (int64_t)gridDim.y);
  const int64_t cbeg = (int64_t)blockIdx.y * cs, cend = cbeg + cs < nchunk ? cbeg + cs : nchunk;
  for (int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); t < N; t += (int64_t)gridDim.x * kWarps) {
    int64_t beg, n;
    if (tok_off) {
      beg = tok_off[t];
      n = tok_off[t + 1] - beg;
    } else {
      beg = t * k;
      n = k;
    }
    const int32_t my_row = lane < n ? tok_rows[beg + lane] : -1;
    // no kept row among the first 32 (token choice: all k; expert choice: the list is
    // non-empty exactly when it has a row, and every listed row is kept)
    const bool pass = x != nullptr && !__any_sync(kFull, my_row >= 0) && (tok_off == nullptr || n == 0);
    for (int64_t c0 = cbeg; c0 < cend; c0 += 32) {
      const int64_t c = c0 + lane;
      const bool act = c < cend;
      float acc[VN];
#pragma unroll
      for (int i = 0; i < VN; ++i) acc[i] = 0.f;
      if (ys && act) {
        const uint4* src = reinterpret_cast<const uint4*>(ys + t * d + c * VN);
#pragma unroll
        for (int q = 0; q < NV; ++q) Vec16<float>::unpack(__ldg(src + q), acc + 4 * q);
      }
      {
        float v[KU][VN];
#pragma unroll
        for (int j = 0; j < KU; ++j) {
          const int32_t row = __shfl_sync(kFull, my_row, j);
          if (act && j < n && row >= 0) {
            const uint4* src = reinterpret_cast<const uint4*>(yp + (int64_t)row * d + c * VN);
#pragma unroll
            for (int q = 0; q < NV; ++q) Vec16<float>::unpack(__ldg(src + q), v[j] + 4 * q);
          } else {
#pragma unroll
            for (int i = 0; i < VN; ++i) v[j][i] = -0.f;  // x + (-0) == x for every x, signed zeros included
          }
        }
#pragma unroll
        for (int j = 0; j < KU; ++j)
#pragma unroll
          for (int i = 0; i < VN; ++i) acc[i] += v[j][i];
      }
      for (int64_t j = KU; j < n; ++j) {
        const int32_t row = j < 32 ? __shfl_sync(kFull, my_row, (int)j) : tok_rows[beg + j];
        if (act && row >= 0) {
          const uint4* src = reinterpret_cast<const uint4*>(yp + (int64_t)row * d + c * VN);
#pragma unroll
          for (int q = 0; q < NV; ++q) {
            float v[4];
            Vec16<float>::unpack(__ldg(src + q), v);
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[4 * q + i] += v[i];
          }
        }
      }
      if (pass && act) {
        float xv[VN];
        VO::unpack(__ldg(reinterpret_cast<const uint4*>(x) + t * nchunk + c), xv);
#pragma unroll
        for (int i = 0; i < VN; ++i) acc[i] += xv[i];
      }
      if (act) reinterpret_cast<uint4*>(out)[t * nchunk + c] = VO::pack(acc);
    }
  }
}

template <typename T>
cudaError_t launch_permute_t(const Plan& p, const void* x, const int32_t* idx, const float* gate, void* xp,
                             int32_t* tok_rows, int32_t* tok_off, int32_t* expert_off, int32_t* row_token,
                             float* row_gate, void* stats, void* ws, cudaStream_t st, PermuteMode mode,
                             const int32_t* shard_counts, int32_t n_shards, int32_t shard_rank) {
  int32_t* status = status_ptr(p, ws);
  int32_t* rank_base = nullptr;
  // MXFP8 experts: the rows go out quantised, scales after the codes (mx::scale_offset)
  uint8_t* xs = p.fp8w && xp ? static_cast<uint8_t*>(xp) + mx::scale_offset(p.max_rows, p.d) : nullptr;
  if (shard_counts) {
    if (p.ec || mode != kCountsFromIdx) return cudaErrorInvalidValue;
    rank_base = ws_at<int32_t>(ws, p.rank_base);
    shard_base_kernel<<<(unsigned)ceil_div(p.E, 256), 256, 0, st>>>(shard_counts, n_shards, shard_rank, p.E,
                                                                    rank_base, status);
  }
  if (p.ec) {
    uint32_t* bits = ws_at<uint32_t>(ws, p.ec_bits);
    cudaError_t err = cudaMemsetAsync(bits, 0, (size_t)(p.N * p.words) * 4, st);
    if (err == cudaSuccess) err = cudaMemsetAsync(tok_off, 0, (size_t)(p.N + 1) * 4, st);
    if (err != cudaSuccess) return err;
    const int64_t n = p.E * p.cap;
    const int64_t nb = ceil_div(n > p.E + 1 ? n : p.E + 1, 256);
    ec_mark_kernel<<<(unsigned)nb, 256, 0, st>>>(idx, gate, p.N, p.E, p.cap, p.words, bits, row_token, row_gate,
                                                 expert_off, tok_off, status);
    ec_tok_scan_kernel<<<1, 1024, 0, st>>>(p.N, p.E, p.cap, tok_off, stats);
    ec_fill_kernel<<<(unsigned)ceil_div(p.N, kWarps), kWarps * 32, 0, st>>>(bits, idx, tok_off, p.N, p.words, p.cap,
                                                                            tok_rows);
    if (xp) {
      const int64_t blocks = ceil_div(p.N, kWarps) < 148 * 16 ? ceil_div(p.N, kWarps) : 148 * 16;
      copy_rows_csr_kernel<T><<<(unsigned)blocks, kWarps * 32, 0, st>>>(static_cast<const T*>(x), tok_rows, tok_off,
                                                                        p.N, p.d, static_cast<T*>(xp), xs);
    }
    return cudaGetLastError();
  }
  int32_t* tile_counts = ws_at<int32_t>(ws, p.tile_counts);
  int32_t* tile_base = ws_at<int32_t>(ws, p.tile_base);
  // row slices per tile so that about two blocks per SM copy rows
  const int64_t nchunk = p.d / (16 / (int64_t)sizeof(T));
  int64_t slices = ceil_div(2 * 148, p.tiles);
  const int64_t max_slices = ceil_div(nchunk, 32);
  if (slices > max_slices) slices = max_slices;
  if (slices < 1 || xp == nullptr) slices = 1;  // (metadata only: one block per tile)
  if (mode == kFusedOffsets) {
    RouterStatsArgs fin{};
    fin.acc = stats_acc_at(ws_at<uint8_t>(ws, p.stat_acc), p.E);
    fin.alpha = p.cfg.aux_alpha;
    const size_t sc_smem = (size_t)p.E * 4 + (size_t)kMaxTileTokens * p.k * 4 + (size_t)(2 * p.E + 1) * 4;
    return launch_pdl(scatter_kernel<T, true>, dim3((unsigned)p.tiles + 1, (unsigned)slices), dim3(kWarps * 32),
                      sc_smem, st, static_cast<const T*>(x), idx, gate, (const int32_t*)tile_counts, expert_off, p.N,
                      p.d, p.k, p.E, (int64_t)p.tiles, p.tile, p.cap, static_cast<T*>(xp), tok_rows, row_token,
                      row_gate, stats, status, fin, (const int32_t*)nullptr, xs);
  }
  if (mode == kCountsFromIdx) {
    const size_t hist_smem = (size_t)kWarps * p.E * 4;
    count_kernel<<<(unsigned)ceil_div(p.tiles, kWarps), kWarps * 32, hist_smem, st>>>(idx, p.N, p.k, p.E, p.tiles,
                                                                                    p.tile, tile_counts, status);
  }
  RouterStatsArgs rs{};
  if (mode == kCountsFromRouter) {
    rs.acc = stats_acc_at(ws_at<uint8_t>(ws, p.stat_acc), p.E);
    rs.alpha = p.cfg.aux_alpha;
  }
  // the router statistics of a sharded batch come from the exchanged partial sums
  if (shard_counts && stats) {
    rs.acc = stats_acc_at(ws_at<uint8_t>(ws, p.stat_acc), p.E);
    rs.alpha = p.cfg.aux_alpha;
  }
  scan_offsets_kernel<<<(unsigned)ceil_div(p.E, kWarps), kWarps * 32, 0, st>>>(
      tile_counts, p.E, p.tiles, p.cap, p.N, p.k, tile_base, expert_off, stats, status + 5, rs, p.Ntot, rank_base);
  const size_t sc_smem = (size_t)p.E * 4 + (size_t)kMaxTileTokens * p.k * 4;
  scatter_kernel<T, false><<<dim3((unsigned)p.tiles, (unsigned)slices), kWarps * 32, sc_smem, st>>>(
      static_cast<const T*>(x), idx, gate, tile_base, expert_off, p.N, p.d, p.k, p.E, p.tiles, p.tile, p.cap,
      static_cast<T*>(xp), tok_rows, row_token, row_gate, stats, status, RouterStatsArgs{}, rank_base, xs);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ec_select(const Plan& p, const float* probs, int32_t* idx, float* gate, float* probs_t,
                             cudaStream_t st) {
  if (probs_t) {  // read each expert's probabilities from an expert-major copy (coalesced)
    ec_transpose_kernel<<<dim3((unsigned)ceil_div(p.N, 32), (unsigned)ceil_div(p.E, 32)), 32 * 8, 0, st>>>(
        probs, p.N, p.E, probs_t);
    ec_select_kernel<<<(unsigned)p.E, 1024, 0, st>>>(probs_t, p.N, 1, p.N, p.E, p.cap, idx, gate);
  } else {
    ec_select_kernel<<<(unsigned)p.E, 1024, 0, st>>>(probs, 1, p.E, p.N, p.E, p.cap, idx, gate);
  }
  return cudaGetLastError();
}

cudaError_t launch_permute(const Plan& p, const void* x, const int32_t* idx, const float* gate, void* xp,
                           int32_t* tok_rows, int32_t* tok_off, int32_t* expert_off, int32_t* row_token,
                           float* row_gate, void* stats, void* ws, cudaStream_t st, PermuteMode mode,
                           const int32_t* shard_counts, int32_t n_shards, int32_t shard_rank) {
  if (p.bf16)
    return launch_permute_t<__nv_bfloat16>(p, x, idx, gate, xp, tok_rows, tok_off, expert_off, row_token, row_gate,
                                           stats, ws, st, mode, shard_counts, n_shards, shard_rank);
  return launch_permute_t<float>(p, x, idx, gate, xp, tok_rows, tok_off, expert_off, row_token, row_gate, stats, ws,
                                 st, mode, shard_counts, n_shards, shard_rank);
}

bool permute_fuses_offsets(const Plan& p) { return !p.ec && p.E * p.tiles <= 8192; }

template <typename... KArgs, typename... Args>
cudaError_t launch_maybe_pdl(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args... args) {
  if (pdl) return launch_pdl(kern, grid, block, smem, st, args...);
  kern<<<grid, block, smem, st>>>(args...);
  return cudaGetLastError();
}

cudaError_t launch_combine(const Plan& p, const void* yp, const int32_t* tok_rows, const int32_t* tok_off,
                           const void* ys, const void* x, void* out, cudaStream_t st, bool pdl) {
  const int64_t blocks = ceil_div(p.N, kWarps) < 148 * 16 ? ceil_div(p.N, kWarps) : 148 * 16;
  const int64_t nchunk = p.d / (p.bf16 ? 8 : 4);
  int64_t slices = ceil_div(4 * 148, blocks);  // small batches: split rows so ~4 blocks per SM combine
  const int64_t max_slices = ceil_div(nchunk, 32);
  if (slices > max_slices) slices = max_slices;
  if (slices < 1) slices = 1;
  const dim3 grid((unsigned)blocks, (unsigned)slices);
  const int32_t* toff = p.ec ? tok_off : nullptr;
  const float* ysf = static_cast<const float*>(ys);
  const float* ypf = static_cast<const float*>(yp);
  // rows loaded together: top-k's k (expert choice: a token has up to E rows, 2 on average for cf 1)
  const int64_t ku = p.ec ? 2 : p.k;
  const __nv_bfloat16* xb = p.passthrough ? static_cast<const __nv_bfloat16*>(x) : nullptr;
  const float* xf = p.passthrough ? static_cast<const float*>(x) : nullptr;
  if (p.bf16) {
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
    if (ku <= 1) launch_maybe_pdl(pdl, combine_kernel<__nv_bfloat16, 1>, grid, dim3(kWarps * 32), 0, st, ypf, (const int32_t*)tok_rows, toff, ysf, p.N, p.d, p.k, o, xb);
    else if (ku <= 2) launch_maybe_pdl(pdl, combine_kernel<__nv_bfloat16, 2>, grid, dim3(kWarps * 32), 0, st, ypf, (const int32_t*)tok_rows, toff, ysf, p.N, p.d, p.k, o, xb);
    else if (ku <= 4) launch_maybe_pdl(pdl, combine_kernel<__nv_bfloat16, 4>, grid, dim3(kWarps * 32), 0, st, ypf, (const int32_t*)tok_rows, toff, ysf, p.N, p.d, p.k, o, xb);
    else launch_maybe_pdl(pdl, combine_kernel<__nv_bfloat16, 8>, grid, dim3(kWarps * 32), 0, st, ypf, (const int32_t*)tok_rows, toff, ysf, p.N, p.d, p.k, o, xb);
  } else {
    float* o = static_cast<float*>(out);
    if (ku <= 1) launch_maybe_pdl(pdl, combine_kernel<float, 1>, grid, dim3(kWarps * 32), 0, st, ypf, (const int32_t*)tok_rows, toff, ysf, p.N, p.d, p.k, o, xf);
    else if (ku <= 2) launch_maybe_pdl(pdl, combine_kernel<float, 2>, grid, dim3(kWarps * 32), 0, st, ypf, (const int32_t*)tok_rows, toff, ysf, p.N, p.d, p.k, o, xf);
    else if (ku <= 4) launch_maybe_pdl(pdl, combine_kernel<float, 4>, grid, dim3(kWarps * 32), 0, st, ypf, (const int32_t*)tok_rows, toff, ysf, p.N, p.d, p.k, o, xf);
    else launch_maybe_pdl(pdl, combine_kernel<float, 8>, grid, dim3(kWarps * 32), 0, st, ypf, (const int32_t*)tok_rows, toff, ysf, p.N, p.d, p.k, o, xf);
  }
  return cudaGetLastError();
}

}  // namespace moe
