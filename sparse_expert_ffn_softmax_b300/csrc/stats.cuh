// Router statistics, accumulated in fixed point so the totals do not depend on
// the order in which blocks finish (integer addition is associative):
//   P_sum[e]  = sum_t p[t,e]         int64, units of 2^-40
//   cnt[e]    = assignments to e     int32
//   lse_sum   = sum_t lse_t          int64, units of 2^-32 (|lse| < 2^16 assumed)
//   lse2_sum  = sum_t lse_t^2        int64, units of 2^-24
// Each router block adds its fp32 block partials (summed over its tokens in a
// fixed order) once. The finaliser computes
//   f_e = cnt_e / total assignments (token choice: before dropping; expert
//         choice: C per expert), P_e = P_sum[e] / N,
//   aux = alpha * E * sum_e f_e P_e, z = (lse_sum / N)^2, mean_lse_sq = lse2_sum / N,
// writes the statistics and zeroes the accumulators for the next call.
// Pages: "Mixture of Experts" (aigrafen.se) auxiliary loss; "Mixture of Experts
// (MoE)" (learn.starphix.com) "Load Balancing (Critical)" (load_balancing_loss, z_loss).
#pragma once

#include "common.cuh"

namespace moe {

constexpr double kPScale = 1099511627776.0;  // 2^40
constexpr double kLseScale = 4294967296.0;   // 2^32
constexpr double kLse2Scale = 16777216.0;    // 2^24

// Accumulator layout (bytes): [P_sum: E x int64][lse_sum, lse2_sum: 2 x int64][cnt: E x int32]
inline __host__ __device__ size_t stats_acc_bytes(int64_t E) { return (size_t)E * 12 + 16; }

struct StatsAcc {
  unsigned long long* p;    // [E]
  unsigned long long* lse;  // [2]
  int32_t* cnt;             // [E]
};
__host__ __device__ inline StatsAcc stats_acc_at(void* base, int64_t E) {
  StatsAcc a;
  a.p = static_cast<unsigned long long*>(base);
  a.lse = a.p + E;
  a.cnt = reinterpret_cast<int32_t*>(a.lse + 2);
  return a;
}

__device__ inline unsigned long long to_fixed(double v, double scale) {
  return static_cast<unsigned long long>(__double2ll_rn(v * scale));
}
__device__ inline double from_fixed(unsigned long long v, double scale) {
  return static_cast<double>(static_cast<long long>(v)) / scale;
}

// Block-wide sum of a double in a fixed order (warp shuffles, then the per-warp
// sums in order). Every thread of the block must call it; all get the sum.
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

// Whole block: statistics from the accumulators, then the accumulators are zeroed.
__device__ inline void finalize_router_stats(StatsAcc acc, int64_t N, int64_t E, int64_t k, int64_t cap, int ec,
                                             float alpha, void* stats) {
  __shared__ double s_warp[32];
  moe_stats_header* hdr = static_cast<moe_stats_header*>(stats);
  float* f_out = reinterpret_cast<float*>(hdr + 1);
  float* P_out = f_out + E;
  int32_t* cnt_out = reinterpret_cast<int32_t*>(P_out + E);
  const double total = ec ? (double)E * (double)cap : (double)N * (double)k;
  double aux_part = 0.0;
  for (int64_t e = threadIdx.x; e < E; e += blockDim.x) {
    const double P = from_fixed(*((volatile unsigned long long*)(acc.p + e)), kPScale) / (double)N;
    const int32_t cnt = ec ? (int32_t)cap : *((volatile int32_t*)(acc.cnt + e));
    const double f = total > 0 ? (double)cnt / total : 0.0;
    f_out[e] = (float)f;
    P_out[e] = (float)P;
    cnt_out[e] = cnt;
    aux_part += f * P;
  }
  const double aux = block_sum_fixed(aux_part, s_warp);
  if (threadIdx.x == 0) {
    const double ml = from_fixed(*((volatile unsigned long long*)(acc.lse)), kLseScale) / (double)N;
    hdr->aux_loss = (float)((double)alpha * (double)E * aux);
    hdr->z_loss = (float)(ml * ml);
    hdr->mean_lse_sq = (float)(from_fixed(*((volatile unsigned long long*)(acc.lse + 1)), kLse2Scale) / (double)N);
    hdr->n_experts = (int32_t)E;
  }
  __syncthreads();  // every read above is done before the reset
  for (int64_t e = threadIdx.x; e < E; e += blockDim.x) {
    acc.p[e] = 0ull;
    acc.cnt[e] = 0;
  }
  if (threadIdx.x == 0) {
    acc.lse[0] = 0ull;
    acc.lse[1] = 0ull;
  }
}

}  // namespace moe
