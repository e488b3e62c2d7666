// Block-level steps of the capacity / dropping computation, shared by the
// router's last block (small layers) and the stand-alone scan kernel:
//  - exclusive prefix of every expert's per-tile assignment counts over the
//    tiles (token order), giving each tile's starting rank per expert;
//  - kept_e = min(count_e, C) and expert_off = exclusive prefix of kept;
//  - the dropping statistics.
// Pages: "Mixture of Experts" (aigrafen.se) "Expert capacity" and its MoE code
// (tokens listed in index order, cut to the first C).
#pragma once

#include "common.cuh"

namespace moe {

// Block-wide exclusive scan for blockDim.x <= 1024 (multiple of 32); returns the
// exclusive prefix of v and writes the block total to *total.
__device__ inline int block_exclusive_scan(int v, int* s_warp /* >= 33 */, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int inc = warp_inclusive_scan(v);
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < nw ? s_warp[lane] : 0;
    const int winc = warp_inclusive_scan(w);
    if (lane < nw) s_warp[lane] = winc - w;
    if (lane == 31) s_warp[32] = winc;
  }
  __syncthreads();
  const int r = s_warp[warp] + inc - v;
  *total = s_warp[32];
  __syncthreads();
  return r;
}

// One warp scans expert e's tile counts [T] into tile_base[e][0..T-1], total at [T].
__device__ inline void scan_expert_tiles(const int32_t* counts, int32_t* base, int64_t T) {
  const int lane = threadIdx.x & 31;
  int carry = 0;
  for (int64_t b = 0; b < T; b += 128) {  // 4 loads in flight per lane
    int v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = b + 32 * u + lane;
      v[u] = i < T ? counts[i] : 0;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = b + 32 * u + lane;
      const int inc = warp_inclusive_scan(v[u]);
      if (i < T) base[i] = carry + inc - v[u];
      carry += __shfl_sync(kFull, inc, 31);
    }
  }
  if (lane == 0) base[T] = carry;
}

// Capacity left to this shard by expert e: C minus the assignments to e in earlier
// shards (rank_base null: the whole batch, C).
__device__ __forceinline__ int64_t cap_left(int64_t cap, const int32_t* rank_base, int64_t e) {
  if (!rank_base) return cap;
  const int64_t c = cap - (int64_t)rank_base[e];
  return c > 0 ? c : 0;
}

// Whole block: offsets over E <= 512 experts from the totals tile_base[e][T],
// and (stats non-null) kept counts and dropping statistics. rank_base (nullable):
// per-expert assignments in earlier shards of a token-sharded batch.
__device__ inline void offsets_from_totals(const int32_t* tile_base, int64_t E, int64_t T, int64_t cap, int64_t N,
                                           int64_t k, int32_t* expert_off, void* stats,
                                           const int32_t* rank_base = nullptr) {
  __shared__ int s_warp[33];
  const int per = (int)ceil_div(E, (int64_t)blockDim.x);  // <= 2 for blockDim >= 256
  const int64_t e0 = (int64_t)threadIdx.x * per;
  int kept[2] = {0, 0}, ksum = 0, dsum = 0;
  for (int i = 0; i < per && i < 2; ++i) {
    const int64_t ee = e0 + i;
    if (ee < E) {
      const int cnt = *((volatile const int32_t*)(tile_base + ee * (T + 1) + T));
      const int64_t cl = cap_left(cap, rank_base, ee);
      kept[i] = (int)(cnt < cl ? cnt : cl);
      ksum += kept[i];
      dsum += cnt - kept[i];
    }
  }
  int rows = 0, dropped = 0;
  int off = block_exclusive_scan(ksum, s_warp, &rows);
  block_exclusive_scan(dsum, s_warp, &dropped);
  for (int i = 0; i < per && i < 2; ++i) {
    const int64_t ee = e0 + i;
    if (ee < E) {
      expert_off[ee] = off;
      off += kept[i];
    }
  }
  if (threadIdx.x == 0) expert_off[E] = rows;
  if (stats) {
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
}

// True in exactly one block: the last of the grid to arrive at the ticket.
// Every thread must call it; the caller's global writes before the call are
// visible to the last block afterwards. The last block resets the ticket.
__device__ inline bool last_block_ticket(int32_t* ticket) {
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(ticket, 1);
    s_last = prev == (int)(gridDim.x * gridDim.y * gridDim.z) - 1;
    if (s_last) *ticket = 0;
  }
  __syncthreads();
  if (s_last) __threadfence();
  return s_last != 0;
}

}  // namespace moe
