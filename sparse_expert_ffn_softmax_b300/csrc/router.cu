// Router: logits = x W_r^T (+ per-expert offset), softmax over experts with its
// log-normaliser, top-k (largest logit first, equal logits to the lower expert
// id), the gate rule, and per-block partial sums for the balancing statistics;
// then a one-block finaliser for f, P, aux loss and z-loss.
//
// Pages: "Mixture of Experts (MoE)" (learn.starphix.com) "Key Equations"
// (router_logits = x @ W_router^T, top-k, weighted combination) and "Load
// Balancing (Critical)" (load_balancing_loss, z_loss); "Mixture of Experts"
// (aigrafen.se) gate formula g = softmax(W_r x), the auxiliary loss
// alpha * N * sum f_i P_i and its MoE code (softmax, topk, renormalise);
// "MoE Architecture" (vanos001.github.io) TokenChoiceRouter (top-k on logits,
// softmax over the k).
//
// One warp per token: the lanes split d into 16-byte vectors and keep one
// partial dot product per expert of the current group of V experts; a
// transpose-reduce (V/2 + ... + 1 shuffles, then a butterfly over the rest)
// leaves lane l with the logit of expert (l mod V). The token's E logits then
// sit in shared memory for the softmax and top-k. Block b owns a fixed range
// of tokens and writes its partial sums in a fixed order, so the statistics
// are deterministic.
#include <cfloat>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kEplMax = 16;  // experts per lane in the softmax / top-k stage: E <= 512

template <int V>
__device__ __forceinline__ void transpose_reduce(float (&a)[V], int lane) {
#pragma unroll
  for (int s = V / 2; s >= 1; s >>= 1) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      float send = upper ? a[i] : a[i + s];
      float keep = upper ? a[i + s] : a[i];
      a[i] = keep + __shfl_xor_sync(kFull, send, s);
    }
  }
#pragma unroll
  for (int s = V; s < 32; s <<= 1) a[0] += __shfl_xor_sync(kFull, a[0], s);
}

struct RouterArgs {
  const void* x;
  const void* wr;
  const float* logit_bias;
  int32_t* idx;
  float* gate;
  float* logits;  // nullable
  float* probs;   // nullable
  float* part_p;      // [E][blocks]
  int32_t* part_cnt;  // [E][blocks]
  float* part_lse;    // [blocks][2]
  int32_t* status;
  int64_t N, d, E, k;
  int gating;
  int tpw;
};

// Dynamic shared memory: [W_r copy (if kWSmem)] [sL: warps x E floats] [sP: warps x E floats] [cnt: E ints]
template <typename T, int V, bool kWSmem>
__global__ void __launch_bounds__(kRouterWarps * 32) router_kernel(RouterArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  using VT = Vec16<T>;
  constexpr int VN = VT::n;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t E = a.E, d = a.d, k = a.k;
  const int64_t nchunk = d / VN;
  const uint4* wsrc = static_cast<const uint4*>(a.wr);
  uint8_t* cur = smem;
  if (kWSmem) {
    uint4* wdst = reinterpret_cast<uint4*>(smem);
    for (int64_t i = threadIdx.x; i < E * nchunk; i += blockDim.x) wdst[i] = wsrc[i];
    wsrc = wdst;
    cur += E * nchunk * 16;
  }
  float* sL = reinterpret_cast<float*>(cur) + warp * E;
  float* sPall = reinterpret_cast<float*>(cur) + kRouterWarps * E;
  int32_t* sCnt = reinterpret_cast<int32_t*>(sPall + kRouterWarps * E);
  for (int64_t e = threadIdx.x; e < E; e += blockDim.x) sCnt[e] = 0;
  __syncthreads();

  float pacc[kEplMax];
#pragma unroll
  for (int i = 0; i < kEplMax; ++i) pacc[i] = 0.f;
  float lse_sum = 0.f, lse_sq = 0.f;
  const bool ec = a.gating == MOE_GATE_EXPERT_CHOICE;

  const int64_t tok0 = (int64_t)blockIdx.x * kRouterWarps * a.tpw + (int64_t)warp * a.tpw;
  for (int it = 0; it < a.tpw; ++it) {
    const int64_t t = tok0 + it;
    if (t >= a.N) break;
    // ---- logits of token t into sL ----
    const uint4* xrow = static_cast<const uint4*>(a.x) + t * nchunk;
    for (int64_t eb = 0; eb < E; eb += V) {
      float acc[V];
#pragma unroll
      for (int v = 0; v < V; ++v) acc[v] = 0.f;
      for (int64_t c = lane; c < nchunk; c += 32) {
        float xv[VN];
        VT::unpack(__ldg(xrow + c), xv);
#pragma unroll
        for (int v = 0; v < V; ++v) {
          if (eb + v < E) {
            float wv[VN];
            uint4 wu = kWSmem ? wsrc[(eb + v) * nchunk + c] : __ldg(wsrc + (eb + v) * nchunk + c);
            VT::unpack(wu, wv);
#pragma unroll
            for (int i = 0; i < VN; ++i) acc[v] = fmaf(xv[i], wv[i], acc[v]);
          }
        }
      }
      transpose_reduce<V>(acc, lane);
      const int64_t e = eb + lane;
      if (lane < V && e < E) sL[e] = acc[0] + (a.logit_bias ? a.logit_bias[e] : 0.f);
    }
    __syncwarp();
    // ---- softmax over experts, log-normaliser ----
    float m = -FLT_MAX;
    for (int64_t e = lane; e < E; e += 32) m = fmaxf(m, sL[e]);
    m = warp_max(m);
    float s = 0.f;
    for (int64_t e = lane; e < E; e += 32) s += expf(sL[e] - m);
    s = warp_sum(s);
    const float lse = m + logf(s);
    if (lane == 0) {
      lse_sum += lse;
      lse_sq += lse * lse;
    }
#pragma unroll
    for (int i = 0; i < kEplMax; ++i) {
      const int64_t e = lane + 32 * i;
      if (e < E) {
        const float L = sL[e];
        const float pe = expf(L - m) / s;
        pacc[i] += pe;
        if (a.probs) a.probs[t * E + e] = pe;
        if (a.logits) a.logits[t * E + e] = L;
      }
    }
    if (!ec) {
      // ---- top-k on logits: repeated warp arg-max, ties to the lower expert id ----
      uint32_t taken = 0;
      int my_e = 0;
      float my_l = 0.f;
      for (int j = 0; j < k; ++j) {
        float bv = -FLT_MAX;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kEplMax; ++i) {
          const int e = lane + 32 * i;
          if (e < E && !((taken >> i) & 1u)) {
            const float v = sL[e];
            if (v > bv || (v == bv && e < be)) {
              bv = v;
              be = e;
            }
          }
        }
#pragma unroll
        for (int sh = 16; sh >= 1; sh >>= 1) {
          const float ov = __shfl_xor_sync(kFull, bv, sh);
          const int oe = __shfl_xor_sync(kFull, be, sh);
          if (ov > bv || (ov == bv && oe < be)) {
            bv = ov;
            be = oe;
          }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (lane == j) {
          my_e = be;
          my_l = bv;
        }
      }
      // ---- gates ----
      float g = 0.f;
      const bool mine = lane < k;
      if (a.gating == MOE_GATE_TOPK_SOFTMAX) {
        const float l0 = __shfl_sync(kFull, my_l, 0);
        const float num = mine ? expf(my_l - l0) : 0.f;
        const float den = warp_sum(num);
        g = num / den;
      } else {
        const float pj = mine ? expf(my_l - m) / s : 0.f;
        if (a.gating == MOE_GATE_SOFTMAX_TOPK_RENORM) {
          const float den = warp_sum(pj);
          g = pj / den;
        } else {
          g = pj;
        }
      }
      if (mine) {
        a.idx[t * k + lane] = my_e;
        a.gate[t * k + lane] = g;
        atomicAdd(&sCnt[my_e], 1);
      }
    }
    __syncwarp();
  }
  // ---- block partials in a fixed order ----
  float* sP = sPall + warp * E;
#pragma unroll
  for (int i = 0; i < kEplMax; ++i) {
    const int64_t e = lane + 32 * i;
    if (e < E) sP[e] = pacc[i];
  }
  __shared__ float sLse[kRouterWarps][2];
  if (lane == 0) {
    sLse[warp][0] = lse_sum;
    sLse[warp][1] = lse_sq;
  }
  __syncthreads();
  for (int64_t e = threadIdx.x; e < E; e += blockDim.x) {
    float acc = 0.f;
    for (int w = 0; w < kRouterWarps; ++w) acc += sPall[w * E + e];
    a.part_p[e * gridDim.x + blockIdx.x] = acc;
    a.part_cnt[e * gridDim.x + blockIdx.x] = sCnt[e];
  }
  if (threadIdx.x == 0) {
    float s0 = 0.f, s1 = 0.f;
    for (int w = 0; w < kRouterWarps; ++w) {
      s0 += sLse[w][0];
      s1 += sLse[w][1];
    }
    a.part_lse[blockIdx.x * 2 + 0] = s0;
    a.part_lse[blockIdx.x * 2 + 1] = s1;
  }
}

// Statistics from the block partials, summed in a fixed order in fp64.
// f_e = count_e / total assignments (token choice: before dropping; expert
// choice: C per expert), P_e = mean_t p[t,e], aux = alpha * E * sum f P,
// z = (mean lse)^2, mean_lse_sq = mean lse^2. Partials are laid out [E][blocks];
// warp w reduces experts w, w+16, ... with its lanes striding over the blocks.
__global__ void __launch_bounds__(512) router_finalize_kernel(const float* part_p, const int32_t* part_cnt,
                                                              const float* part_lse, int64_t blocks, int64_t N,
                                                              int64_t E, int64_t k, int64_t cap, int ec,
                                                              float alpha, void* stats) {
  __shared__ double red[3][512];
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
  red[0][threadIdx.x] = aux_part;
  red[1][threadIdx.x] = l0;
  red[2][threadIdx.x] = l1;
  __syncthreads();
  for (int s = 256; s >= 1; s >>= 1) {
    if ((int)threadIdx.x < s) {
#pragma unroll
      for (int q = 0; q < 3; ++q) red[q][threadIdx.x] += red[q][threadIdx.x + s];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double ml = red[1][0] / (double)N;
    hdr->aux_loss = (float)((double)alpha * (double)E * red[0][0]);
    hdr->z_loss = (float)(ml * ml);
    hdr->mean_lse_sq = (float)(red[2][0] / (double)N);
    hdr->n_experts = (int32_t)E;
  }
}

template <typename T, int V, bool kWSmem>
cudaError_t launch_router_t(const Plan& p, RouterArgs a, cudaStream_t st) {
  const size_t wbytes = kWSmem ? (size_t)(p.E * p.d * sizeof(T)) : 0;
  const size_t smem = wbytes + (size_t)(2 * kRouterWarps * p.E) * 4 + (size_t)p.E * 4;
  auto kern = router_kernel<T, V, kWSmem>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  kern<<<(unsigned)p.router_blocks, kRouterWarps * 32, smem, st>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_router_dt(const Plan& p, RouterArgs a, cudaStream_t st) {
  const bool wsm = (size_t)(p.E * p.d * sizeof(T)) <= 96 * 1024;
  if (p.E <= 8) return wsm ? launch_router_t<T, 8, true>(p, a, st) : launch_router_t<T, 8, false>(p, a, st);
  if (p.E <= 16) return wsm ? launch_router_t<T, 16, true>(p, a, st) : launch_router_t<T, 16, false>(p, a, st);
  return wsm ? launch_router_t<T, 32, true>(p, a, st) : launch_router_t<T, 32, false>(p, a, st);
}

}  // namespace

cudaError_t launch_router(const Plan& p, const void* x, const moe_weights* w, int32_t* idx, float* gate,
                          float* logits, float* probs, void* stats, void* ws, cudaStream_t st) {
  RouterArgs a;
  a.x = x;
  a.wr = w->w_router;
  a.logit_bias = w->logit_bias;
  a.idx = idx;
  a.gate = gate;
  a.logits = logits;
  a.probs = probs;
  a.part_p = ws_at<float>(ws, p.part_p);
  a.part_cnt = ws_at<int32_t>(ws, p.part_cnt);
  a.part_lse = ws_at<float>(ws, p.part_lse);
  a.status = status_ptr(p, ws);
  a.N = p.N;
  a.d = p.d;
  a.E = p.E;
  a.k = p.k;
  a.gating = p.cfg.gating;
  a.tpw = p.router_tpw;
  cudaError_t err = p.bf16 ? launch_router_dt<__nv_bfloat16>(p, a, st) : launch_router_dt<float>(p, a, st);
  if (err != cudaSuccess) return err;
  router_finalize_kernel<<<1, 512, 0, st>>>(a.part_p, a.part_cnt, a.part_lse, p.router_blocks, p.N, p.E, p.k,
                                            p.cap, p.ec ? 1 : 0, p.cfg.aux_alpha, stats);
  return cudaGetLastError();
}

}  // namespace moe
