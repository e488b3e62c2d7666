// Router statistics from per-block partial sums, reduced by one thread block in
// a fixed order (fp64), so the result does not depend on scheduling.
//   f_e = count_e / total assignments (token choice: before dropping; expert
//         choice: C per expert), P_e = mean_t p[t,e],
//   aux = alpha * E * sum_e f_e P_e, z = (mean_t lse_t)^2, mean_lse_sq = mean_t lse_t^2.
// Pages: "Mixture of Experts" (aigrafen.se) auxiliary loss; "Mixture of Experts
// (MoE)" (learn.starphix.com) "Load Balancing (Critical)" (load_balancing_loss, z_loss).
#pragma once

#include "common.cuh"

namespace moe {

// Block-wide sum of a double in a fixed order (warp shuffles, then warp 0 over
// the per-warp sums). Every thread of the block must call it; all get the sum.
__device__ inline double block_sum_fixed(double v, double* s_warp /* >= 32 */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) v += __shfl_xor_sync(kFull, v, s);
  __syncthreads();
  if (lane == 0) s_warp[warp] = v;
  __syncthreads();
  double t = 0.0;
  for (int w = 0; w < nw; ++w) t += s_warp[w];
  __syncthreads();
  return t;
}

// part_p / part_cnt are [E][blocks], part_lse is [blocks][2].
__device__ inline void finalize_router_stats(const float* part_p, const int32_t* part_cnt, const float* part_lse,
                                             int64_t blocks, int64_t N, int64_t E, int64_t k, int64_t cap, int ec,
                                             float alpha, void* stats) {
  __shared__ double s_warp[32];
  moe_stats_header* hdr = static_cast<moe_stats_header*>(stats);
  float* f_out = reinterpret_cast<float*>(hdr + 1);
  float* P_out = f_out + E;
  int32_t* cnt_out = reinterpret_cast<int32_t*>(P_out + E);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const double total = ec ? (double)E * (double)cap : (double)N * (double)k;
  double aux_part = 0.0;
  for (int64_t e = warp; e < E; e += nwarps) {
    double P = 0.0;
    long long cnt = 0;
#pragma unroll 4
    for (int64_t b = lane; b < blocks; b += 32) {
      P += part_p[e * blocks + b];
      cnt += part_cnt[e * blocks + b];
    }
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
      P += __shfl_xor_sync(kFull, P, s);
      cnt += __shfl_xor_sync(kFull, cnt, s);
    }
    if (ec) cnt = cap;
    P /= (double)N;
    const double f = total > 0 ? (double)cnt / total : 0.0;
    if (lane == 0) {
      f_out[e] = (float)f;
      P_out[e] = (float)P;
      cnt_out[e] = (int32_t)cnt;
      aux_part += f * P;
    }
  }
  double l0 = 0.0, l1 = 0.0;
  for (int64_t b = threadIdx.x; b < blocks; b += blockDim.x) {
    l0 += part_lse[2 * b];
    l1 += part_lse[2 * b + 1];
  }
  const double aux = block_sum_fixed(aux_part, s_warp);
  const double ls = block_sum_fixed(l0, s_warp);
  const double ls2 = block_sum_fixed(l1, s_warp);
  if (threadIdx.x == 0) {
    const double ml = ls / (double)N;
    hdr->aux_loss = (float)((double)alpha * (double)E * aux);
    hdr->z_loss = (float)(ml * ml);
    hdr->mean_lse_sq = (float)(ls2 / (double)N);
    hdr->n_experts = (int32_t)E;
  }
}

}  // namespace moe
