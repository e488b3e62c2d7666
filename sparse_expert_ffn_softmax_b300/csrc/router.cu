// Router: logits = x W_r^T (+ per-expert offset), softmax over experts with its
// log-normaliser, top-k (largest logit first, equal logits to the lower expert
// id), the gate rule, and per-block partial sums for the balancing statistics.
//
// Pages: "Mixture of Experts (MoE)" (learn.starphix.com) "Key Equations"
// (router_logits = x @ W_router^T, top-k, weighted combination) and "Load
// Balancing (Critical)" (load_balancing_loss, z_loss); "Mixture of Experts"
// (aigrafen.se) gate formula g = softmax(W_r x), the auxiliary loss
// alpha * N * sum f_i P_i and its MoE code (softmax, topk, renormalise);
// "MoE Architecture" (vanos001.github.io) TokenChoiceRouter (top-k on logits,
// softmax over the k).
//
// One block = one tile of 8, 16 or 32 consecutive tokens, one warp per token
// (8 warps, 1-4 tokens each). Lane l keeps the logits of experts l, l+32, ... in registers.
// For E <= 32 the lanes split d into 16-byte vectors and keep one partial dot
// product per expert of a group of V experts; a transpose-reduce (V/2 + ... + 1
// shuffles, then a butterfly over the rest) leaves lane l with the logit of
// expert (l mod V). For more experts (bf16) the logits come from the
// tensor-core GEMM (gemm_tc.cu). Each block writes its partial sums in a fixed
// order and adds them to fixed-point accumulators, so the statistics are
// deterministic; a later kernel (the permute's, or router_finalize_kernel) turns
// them into the statistics.
#include <cfloat>

#include "common.cuh"
#include "internal.h"
#include "stats.cuh"

namespace moe {
namespace {

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
  const float* logits_in;  // non-null: fp32 logits [N, E] (bias included) or, splits > 1,
                           // [splits][N, E] partial sums without the bias
  int64_t splits, part_stride;  // slabs of logits_in and the elements between them
  int32_t* idx;
  float* gate;
  float* logits;  // nullable
  float* probs;   // nullable
  StatsAcc acc;       // fixed-point statistic accumulators (stats.cuh)
  int32_t* tile_counts;  // [E][blocks] per-tile assignment counts for the permute, or null
  int32_t* status;
  int64_t N, d, E, k, cap, tile;
  int gating;
  float alpha;
};

// Dynamic shared memory: [W_r copy (kWSmem)] [sP: 8 warps x E] [cnt: E].
// EPL = experts per lane (ceil(E / 32)); V = experts per dot-product group.
template <typename T, int V, int CPL, int EPL, bool kWSmem, bool kLogitsIn>
__global__ void __launch_bounds__(kRouterWarps * 32) router_kernel(RouterArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  using VT = Vec16<T>;
  constexpr int VN = VT::n;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t E = a.E, d = a.d, k = a.k;
  const int64_t nchunk = d / VN;
  const uint4* wsrc = static_cast<const uint4*>(a.wr);
  float* wsm = reinterpret_cast<float*>(smem);  // kWSmem: W_r widened to fp32, [E][d]
  uint8_t* cur = smem;
  if (kWSmem) {
    // stage W_r as fp32 with 8 loads in flight per thread
    const int64_t n = E * nchunk;
    for (int64_t i0 = threadIdx.x; i0 < n; i0 += (int64_t)blockDim.x * 8) {
      uint4 tmp[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t i = i0 + (int64_t)u * blockDim.x;
        if (i < n) tmp[u] = __ldg(wsrc + i);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t i = i0 + (int64_t)u * blockDim.x;
        if (i < n) {
          float f[VN];
          VT::unpack(tmp[u], f);
          float4* dst = reinterpret_cast<float4*>(wsm + i * VN);
#pragma unroll
          for (int q = 0; q < VN / 4; ++q) dst[q] = make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
        }
      }
    }
    cur += E * d * 4;
  }
  float* sPall = reinterpret_cast<float*>(cur);
  int32_t* sCnt = reinterpret_cast<int32_t*>(sPall + kRouterWarps * E);
  for (int64_t e = threadIdx.x; e < E; e += blockDim.x) sCnt[e] = 0;
  __syncthreads();

  float pacc[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) pacc[i] = 0.f;
  float lse_sum = 0.f, lse_sq = 0.f;
  const bool ec = a.gating == MOE_GATE_EXPERT_CHOICE;

  for (int64_t it = 0; it < a.tile / kRouterWarps; ++it) {
    const int64_t t = (int64_t)blockIdx.x * a.tile + it * kRouterWarps + warp;
    if (t >= a.N) break;
    // ---- logits of token t: lane l holds expert l + 32 i in Lr[i] ----
    float Lr[EPL];
    if (kLogitsIn) {
      // the lane's experts' logits: one slab, or K-split slabs added in slab order (the
      // loads of two slabs in flight together, then their two additions in order)
      const float* src = a.logits_in + t * E;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int64_t e = lane + 32 * i;
        Lr[i] = e < E ? src[e] : 0.f;  // (one slab: bias included)
      }
      int64_t sp = 1;
      for (; sp + 1 < a.splits; sp += 2) {
        float v[2][EPL];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int i = 0; i < EPL; ++i) {
            const int64_t e = lane + 32 * i;
            v[u][i] = e < E ? src[(sp + u) * a.part_stride + e] : 0.f;
          }
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int i = 0; i < EPL; ++i) Lr[i] += v[u][i];
      }
      for (; sp < a.splits; ++sp) {
        float v[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          const int64_t e = lane + 32 * i;
          v[i] = e < E ? src[sp * a.part_stride + e] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < EPL; ++i) Lr[i] += v[i];
      }
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int64_t e = lane + 32 * i;
        if (a.splits > 1 && a.logit_bias && e < E) Lr[i] += a.logit_bias[e];
        if (e >= E) Lr[i] = -FLT_MAX;
      }
    } else {
      const uint4* xrow = static_cast<const uint4*>(a.x) + t * nchunk;
#pragma unroll
      for (int gi = 0; gi < EPL; ++gi) {
        // experts eb .. eb+V-1 (V = 32 whenever EPL > 1)
        const int64_t eb = (int64_t)gi * 32;
        float acc[V];
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = 0.f;
        for (int64_t cb = 0; cb < nchunk; cb += CPL * 32) {
          uint4 xr[CPL];
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            const int64_t c = cb + lane + 32 * i;
            xr[i] = c < nchunk ? __ldg(xrow + c) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            const int64_t c = cb + lane + 32 * i;
            if (c < nchunk) {
              float xv[VN];
              VT::unpack(xr[i], xv);
#pragma unroll
              for (int v = 0; v < V; ++v) {
                if (eb + v < E) {
                  float wv[VN];
                  if (kWSmem) {
                    const float4* wp = reinterpret_cast<const float4*>(wsm + ((eb + v) * nchunk + c) * VN);
#pragma unroll
                    for (int q = 0; q < VN / 4; ++q) {
                      const float4 w4 = wp[q];
                      wv[4 * q] = w4.x;
                      wv[4 * q + 1] = w4.y;
                      wv[4 * q + 2] = w4.z;
                      wv[4 * q + 3] = w4.w;
                    }
                  } else {
                    VT::unpack(__ldg(wsrc + (eb + v) * nchunk + c), wv);
                  }
#pragma unroll
                  for (int q = 0; q < VN; ++q) acc[v] = fmaf(xv[q], wv[q], acc[v]);
                }
              }
            }
          }
        }
        transpose_reduce<V>(acc, lane);  // lane l: expert eb + (l mod V)
        const int64_t e = eb + lane;
        Lr[gi] = (lane < V && e < E) ? acc[0] + (a.logit_bias ? a.logit_bias[e] : 0.f) : -FLT_MAX;
      }
    }
    // ---- softmax over experts, log-normaliser ----
    float m = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < EPL; ++i) m = fmaxf(m, Lr[i]);
    m = warp_max(m);
    float ex[EPL];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      ex[i] = lane + 32 * i < E ? __expf(Lr[i] - m) : 0.f;
      s += ex[i];
    }
    s = warp_sum(s);
    const float lse = m + __logf(s);
    const float inv_s = __fdividef(1.f, s);
    if (lane == 0) {
      // explicit roundings: the same sums whichever outputs a call stores (a contracted
      // multiply-add would round once, and the compiler may contract it in one
      // specialisation of the loop and not in another)
      lse_sum = __fadd_rn(lse_sum, lse);
      lse_sq = __fadd_rn(lse_sq, __fmul_rn(lse, lse));
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int64_t e = lane + 32 * i;
      if (e < E) {
        const float pe = __fmul_rn(ex[i], inv_s);
        pacc[i] = __fadd_rn(pacc[i], pe);
        if (a.probs) a.probs[t * E + e] = pe;
        if (a.logits) a.logits[t * E + e] = Lr[i];
      }
    }
    if (!ec) {
      // ---- top-k on logits: repeated warp arg-max, ties to the lower expert id ----
      // Logits as order-preserving unsigned keys (flip the sign bit of positives, all
      // bits of negatives; -0 as +0; a taken or absent expert has key 0): a round is the lane's
      // best key (ascending i, so the lower id on ties), one warp max-reduction of the
      // keys and one min-reduction of the ids holding that key.
      uint32_t key[EPL];
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const uint32_t u = __float_as_uint(Lr[i]) & (Lr[i] == 0.f ? 0u : 0xFFFFFFFFu);  // -0 ties with +0
        key[i] = lane + 32 * i < E ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;
      }
      int my_e = 0;
      float my_l = 0.f;
      for (int j = 0; j < k; ++j) {
        uint32_t bk = key[0];
        int bi = 0;
#pragma unroll
        for (int i = 1; i < EPL; ++i)
          if (key[i] > bk) {
            bk = key[i];
            bi = i;
          }
        const uint32_t mk = __reduce_max_sync(kFull, bk);
        const uint32_t be = __reduce_min_sync(kFull, bk == mk ? (uint32_t)(lane + 32 * bi) : 0xFFFFFFFFu);
        if ((int)(be & 31) == lane) {
#pragma unroll
          for (int i = 0; i < EPL; ++i)
            if (i == (int)(be >> 5)) key[i] = 0u;
        }
        if (lane == j) {
          my_e = (int)be;
          my_l = __uint_as_float((mk & 0x80000000u) ? (mk & 0x7FFFFFFFu) : ~mk);
        }
      }
      // ---- gates ----
      float g = 0.f;
      const bool mine = lane < k;
      if (a.gating == MOE_GATE_TOPK_SOFTMAX) {
        const float l0 = __shfl_sync(kFull, my_l, 0);
        const float num = mine ? __expf(my_l - l0) : 0.f;
        const float den = warp_sum(num);
        g = __fdividef(num, den);
      } else {
        const float pj = mine ? __expf(my_l - m) * inv_s : 0.f;
        if (a.gating == MOE_GATE_SOFTMAX_TOPK_RENORM) {
          const float den = warp_sum(pj);
          g = __fdividef(pj, den);
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
  }
  // ---- block partials in a fixed order ----
  float* sP = sPall + warp * E;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
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
    atomicAdd(a.acc.p + e, to_fixed((double)acc, kPScale));
    if (sCnt[e]) atomicAdd(a.acc.cnt + e, sCnt[e]);
    if (a.tile_counts) a.tile_counts[e * gridDim.x + blockIdx.x] = sCnt[e];
  }
  if (threadIdx.x == 0) {
    float s0 = 0.f, s1 = 0.f;
    for (int w = 0; w < kRouterWarps; ++w) {
      s0 += sLse[w][0];
      s1 += sLse[w][1];
    }
    atomicAdd(a.acc.lse, to_fixed((double)s0, kLseScale));
    atomicAdd(a.acc.lse + 1, to_fixed((double)s1, kLse2Scale));
  }
}


// ---- router for bf16 layers with up to 32 experts: warp-level tensor-core MMAs ----
// A 16-token group of the batch is one m16 tile; the router's E <= 32 rows are up to
// four n8 tiles. KS warps share a group (4; 16 for batches of fewer groups than
// SMs), each taking every KS-th 32-deep slice of K: thread (gid = lane / 4, tig = lane % 4) loads 16 bytes of
// token rows gid and gid + 8 and of router row gid of each n-tile at columns
// 8 tig .. 8 tig + 7 of the slice, which feeds two m16n8k16 MMAs. (The order of
// the K positions inside a slice is the same permutation for both operands, so
// the dot products are unchanged.) The partial accumulators of the warps are
// added in warp order through shared memory, then the group's first warp routes:
// the four lanes of a quad hold the E logits of tokens gid and gid + 8, so the
// softmax, the top-k (larger logit first, equal logits by lower expert id) and
// the gate rule take two shuffle rounds per reduction. Statistics: probability
// sums per expert and lse sums added to the fixed-point accumulators once per
// group; assignment counts per permute tile through shared memory.
__device__ __forceinline__ void mma_16816_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// NT n8 tiles (E <= 8 NT), top-k lists of up to KMAX, KS warps per group; G
// 16-token groups per block (blockDim = 32 KS G, G <= 2, G = 1 for KS = 16);
// TB = 16 G tokens per block = a whole number of permute tiles of a.tile tokens.
template <int NT, int KMAX, int KS>
__global__ void __launch_bounds__(KS == 16 ? 512 : 256, KS == 16 ? 1 : 2) router_mma_kernel(RouterArgs a) {
  constexpr int NV = 2 * NT;  // logits per thread and token
  constexpr int kMmaKSplit = KS;
  __shared__ float s_red[KS == 16 ? 1 : 2][KS][NT * 4][32];
  __shared__ int32_t s_cnt[2][32];  // per permute tile of the block (at most 2) and expert
  pdl_wait();
  pdl_launch_next();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int G = (int)(blockDim.x / (32 * kMmaKSplit));
  const int grp = warp / kMmaKSplit, ks = warp % kMmaKSplit;
  const int gid = lane >> 2, tig = lane & 3;
  const int64_t N = a.N, E = a.E, d = a.d, k = a.k, TT = a.tile;
  const int64_t TB = 16 * (int64_t)G;
  const int64_t blk_t0 = (int64_t)blockIdx.x * TB;
  const int64_t t0 = blk_t0 + grp * 16;
  const int64_t r0 = t0 + gid, r1 = t0 + gid + 8;
  const bool v0 = r0 < N, v1 = r1 < N;
  const bool ec = a.gating == MOE_GATE_EXPERT_CHOICE;
  for (int i = threadIdx.x; i < 2 * 32; i += blockDim.x) (&s_cnt[0][0])[i] = 0;

  // ---- logits: this warp's K slices ----
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);
  const __nv_bfloat16* wr = static_cast<const __nv_bfloat16*>(a.wr);
  const __nv_bfloat16* xr0 = x + (v0 ? r0 : 0) * d + tig * 8;
  const __nv_bfloat16* xr1 = x + (v1 ? r1 : 0) * d + tig * 8;
  float c[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.f;
  const int64_t kslices = d / 32;
#pragma unroll 4
  for (int64_t kb = ks; kb < kslices; kb += kMmaKSplit) {
    const int64_t col = kb * 32;
    const uint4 xa = v0 ? __ldg(reinterpret_cast<const uint4*>(xr0 + col)) : make_uint4(0, 0, 0, 0);
    const uint4 xb = v1 ? __ldg(reinterpret_cast<const uint4*>(xr1 + col)) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int64_t e = 8 * j + gid;
      const uint4 w = e < E ? __ldg(reinterpret_cast<const uint4*>(wr + e * d + col + tig * 8)) : make_uint4(0, 0, 0, 0);
      mma_16816_bf16(c[j], xa.x, xb.x, xa.y, xb.y, w.x, w.y);
      mma_16816_bf16(c[j], xa.z, xb.z, xa.w, xb.w, w.z, w.w);
    }
  }
  // ---- add the K-split partials in warp order ----
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int q = 0; q < 4; ++q) s_red[grp][ks][4 * j + q][lane] = c[j][q];
  __syncthreads();
  if (ks == 0) {
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float v = s_red[grp][0][4 * j + q][lane];
#pragma unroll
        for (int w = 1; w < kMmaKSplit; ++w) v += s_red[grp][w][4 * j + q][lane];
        c[j][q] = v;
      }
    // ---- route tokens gid (h = 0) and gid + 8 (h = 1) ----
    float pacc[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) pacc[i] = 0.f;
    float lse_sum = 0.f, lse_sq = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t t = h ? r1 : r0;
      const bool valid = h ? v1 : v0;
      float L[NV];
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int64_t e = 8 * (i >> 1) + 2 * tig + (i & 1);
        L[i] = e < E ? c[i >> 1][2 * h + (i & 1)] + (a.logit_bias ? a.logit_bias[e] : 0.f) : -FLT_MAX;
      }
      float m = -FLT_MAX;
#pragma unroll
      for (int i = 0; i < NV; ++i) m = fmaxf(m, L[i]);
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 2));
      float ex[NV];
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int64_t e = 8 * (i >> 1) + 2 * tig + (i & 1);
        ex[i] = e < E ? __expf(L[i] - m) : 0.f;
        s += ex[i];
      }
      s += __shfl_xor_sync(kFull, s, 1);
      s += __shfl_xor_sync(kFull, s, 2);
      const float lse = m + __logf(s);
      const float inv_s = __fdividef(1.f, s);
      if (valid && tig == 0) {
        lse_sum = __fadd_rn(lse_sum, lse);  // explicit roundings, as in router_kernel
        lse_sq = __fadd_rn(lse_sq, __fmul_rn(lse, lse));
      }
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int64_t e = 8 * (i >> 1) + 2 * tig + (i & 1);
        if (valid && e < E) {
          const float pe = __fmul_rn(ex[i], inv_s);
          pacc[i] = __fadd_rn(pacc[i], pe);
          if (a.probs) a.probs[t * E + e] = pe;
          if (a.logits) a.logits[t * E + e] = L[i];
        }
      }
      if (!ec) {
        // ---- top-k: repeated quad arg-max, ties to the lower expert id ----
        uint32_t taken = 0;
        float topv[KMAX];
        int topi[KMAX];
#pragma unroll
        for (int r = 0; r < KMAX; ++r) {
          topv[r] = -FLT_MAX;
          topi[r] = 0x7fffffff;
          if (r < k) {
            float bv = -FLT_MAX;
            int be = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
              const int e = 8 * (i >> 1) + 2 * tig + (i & 1);
              if (e < E && !((taken >> i) & 1u) && (L[i] > bv || (L[i] == bv && e < be))) {
                bv = L[i];
                be = e;
              }
            }
#pragma unroll
            for (int sh = 1; sh <= 2; sh <<= 1) {
              const float ov = __shfl_xor_sync(kFull, bv, sh);
              const int oe = __shfl_xor_sync(kFull, be, sh);
              if (ov > bv || (ov == bv && oe < be)) {
                bv = ov;
                be = oe;
              }
            }
#pragma unroll
            for (int i = 0; i < NV; ++i)
              if (8 * (i >> 1) + 2 * tig + (i & 1) == be) taken |= 1u << i;
            topv[r] = bv;
            topi[r] = be;
          }
        }
        // ---- gates ----
        float g[KMAX];
        float den = 0.f;
#pragma unroll
        for (int r = 0; r < KMAX; ++r) {
          g[r] = 0.f;
          if (r < k) {
            g[r] = a.gating == MOE_GATE_TOPK_SOFTMAX ? __expf(topv[r] - topv[0]) : __expf(topv[r] - m) * inv_s;
            den += g[r];
          }
        }
        const bool renorm = a.gating == MOE_GATE_TOPK_SOFTMAX || a.gating == MOE_GATE_SOFTMAX_TOPK_RENORM;
        const float ginv = renorm ? __fdividef(1.f, den) : 1.f;
        if (valid && tig == 0) {
          const int tl = (int)((t - blk_t0) / TT);
#pragma unroll
          for (int r = 0; r < KMAX; ++r)
            if (r < k) {
              a.idx[t * k + r] = topi[r];
              a.gate[t * k + r] = g[r] * ginv;
              if ((unsigned)topi[r] < (unsigned)E) atomicAdd(&s_cnt[tl][topi[r]], 1);
            }
        }
      }
    }
    // ---- statistics of this group: probability sums per expert, lse sums ----
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      float v = pacc[i];
      v += __shfl_xor_sync(kFull, v, 4);
      v += __shfl_xor_sync(kFull, v, 8);
      v += __shfl_xor_sync(kFull, v, 16);
      const int64_t e = 8 * (i >> 1) + 2 * tig + (i & 1);
      if (gid == 0 && e < E) atomicAdd(a.acc.p + e, to_fixed((double)v, kPScale));
    }
    const float l1 = warp_sum(lse_sum), l2 = warp_sum(lse_sq);
    if (lane == 0) {
      atomicAdd(a.acc.lse, to_fixed((double)l1, kLseScale));
      atomicAdd(a.acc.lse + 1, to_fixed((double)l2, kLse2Scale));
    }
  }
  __syncthreads();
  // ---- complete per-tile assignment counts ----
  if (!ec) {
    const int ntl = (int)(TB / TT);
    for (int i = threadIdx.x; i < ntl * E; i += blockDim.x) {
      const int tl = i / (int)E, e = i - tl * (int)E;
      const int64_t tile = (int64_t)blockIdx.x * ntl + tl;
      const int cnt = s_cnt[tl][e];
      if (a.tile_counts && tile * TT < N) a.tile_counts[(int64_t)e * ((N + TT - 1) / TT) + tile] = cnt;
      if (cnt) atomicAdd(a.acc.cnt + e, cnt);
    }
  }
}

}  // namespace

__global__ void __launch_bounds__(512) router_finalize_kernel(StatsAcc acc, int64_t N, int64_t E, int64_t k,
                                                              int64_t cap, int ec, float alpha, void* stats) {
  finalize_router_stats(acc, N, E, k, cap, ec, alpha, stats);
}

namespace {

template <typename T, int V, int CPL, int EPL, bool kWSmem, bool kLogitsIn>
cudaError_t launch_router_t(const Plan& p, RouterArgs a, cudaStream_t st) {
  const size_t wbytes = kWSmem ? (size_t)(p.E * p.d * 4) : 0;
  const size_t smem = wbytes + (size_t)(kRouterWarps * p.E) * 4 + (size_t)p.E * 4;
  auto kern = router_kernel<T, V, CPL, EPL, kWSmem, kLogitsIn>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  kern<<<(unsigned)p.tiles, kRouterWarps * 32, smem, st>>>(a);
  return cudaGetLastError();
}

template <typename T, int V, int CPL, int EPL>
cudaError_t launch_router_w(const Plan& p, RouterArgs a, cudaStream_t st) {
  const bool wsm = (size_t)(p.E * p.d * 4) <= 128 * 1024;
  return wsm ? launch_router_t<T, V, CPL, EPL, true, false>(p, a, st)
             : launch_router_t<T, V, CPL, EPL, false, false>(p, a, st);
}

// CPL: 16-byte chunks of the token row each lane holds at once (the loop over
// the row covers any d). Layers with more than 64 experts, whose unrolled dot
// products are long already, take the shortest, which keeps the number of
// instantiations (and the build time) small.
template <typename T, int V, int EPL>
cudaError_t launch_router_c(const Plan& p, RouterArgs a, cudaStream_t st) {
  const int64_t cpl = ceil_div(p.d / (16 / (int64_t)sizeof(T)), 32);
  if constexpr (EPL > 2) {
    return launch_router_w<T, V, 2, EPL>(p, a, st);
  } else {
    if (cpl <= 2) return launch_router_w<T, V, 2, EPL>(p, a, st);
    if (cpl <= 4) return launch_router_w<T, V, 4, EPL>(p, a, st);
    if (cpl <= 8) return launch_router_w<T, V, 8, EPL>(p, a, st);
    return launch_router_w<T, V, 16, EPL>(p, a, st);
  }
}

template <typename T>
cudaError_t launch_router_logits_in(const Plan& p, RouterArgs a, cudaStream_t st) {
  if (p.E <= 32) return launch_router_t<T, 32, 1, 1, false, true>(p, a, st);
  if (p.E <= 64) return launch_router_t<T, 32, 1, 2, false, true>(p, a, st);
  if (p.E <= 128) return launch_router_t<T, 32, 1, 4, false, true>(p, a, st);
  if (p.E <= 256) return launch_router_t<T, 32, 1, 8, false, true>(p, a, st);
  return launch_router_t<T, 32, 1, 16, false, true>(p, a, st);
}

template <typename T>
cudaError_t launch_router_simt(const Plan& p, RouterArgs a, cudaStream_t st) {
  if (p.E <= 8) return launch_router_c<T, 8, 1>(p, a, st);
  if (p.E <= 16) return launch_router_c<T, 16, 1>(p, a, st);
  if (p.E <= 32) return launch_router_c<T, 32, 1>(p, a, st);
  if constexpr (sizeof(T) == 2) {
    return cudaErrorInvalidValue;  // bf16 layers with E > 32 route from tensor-core logits
  } else {
    if (p.E <= 64) return launch_router_c<T, 32, 2>(p, a, st);
    if (p.E <= 128) return launch_router_c<T, 32, 4>(p, a, st);
    if (p.E <= 256) return launch_router_c<T, 32, 8>(p, a, st);
    return launch_router_c<T, 32, 16>(p, a, st);
  }
}

}  // namespace

template <int NT, int KMAX>
cudaError_t launch_router_mma_t(const Plan& p, RouterArgs a, cudaStream_t st) {
  const int G = p.tile >= 32 ? 2 : 1;  // a block routes a whole number of permute tiles
  const int64_t TB = 16 * G;
  const int64_t blocks = ceil_div(p.N, TB);
  // few groups in the batch: more warps split each group's K range (decided on the whole
  // batch, so a shard sums its logits in the same order as the unsharded batch)
  if (G == 1 && ceil_div(p.Ntot, TB) < 148) {
    return launch_pdl(router_mma_kernel<NT, KMAX, 16>, dim3((unsigned)blocks), dim3(32 * 16), 0, st, a);
  }
  return launch_pdl(router_mma_kernel<NT, KMAX, 4>, dim3((unsigned)blocks), dim3(32 * 4 * G), 0, st, a);
}

template <int KMAX>
cudaError_t launch_router_mma_k(const Plan& p, RouterArgs a, cudaStream_t st) {
  if (p.E <= 8) return launch_router_mma_t<1, KMAX>(p, a, st);
  if (p.E <= 16) return launch_router_mma_t<2, KMAX>(p, a, st);
  if (p.E <= 24) return launch_router_mma_t<3, KMAX>(p, a, st);
  return launch_router_mma_t<4, KMAX>(p, a, st);
}

// bf16 layers with up to 32 experts and k <= 8 (expert choice: any k).
bool router_uses_mma(const Plan& p) { return p.bf16 && p.E <= 32 && (p.ec || p.k <= 8) && p.d % 32 == 0; }

// Router per layer shape:
//  - bf16 with more than 32 experts: the tensor cores write the logits (K split
//    for small batches, router_k_splits), then this file's kernel routes;
//  - bf16 layers with up to 32 experts: router_mma_kernel (warp-level tensor-core
//    MMAs on 16-token tiles, routing by lane quads);
//  - fp32 layers (and bf16 with k > 8): the SIMT router (dot products on the CUDA
//    cores, one warp per token).
bool router_uses_tc(const Plan& p) { return p.bf16 && p.E >= kRouterTcMinE; }

cudaError_t launch_router_stats_finalize(const Plan& p, void* ws, void* stats, cudaStream_t st) {
  router_finalize_kernel<<<1, 512, 0, st>>>(stats_acc_at(ws_at<uint8_t>(ws, p.stat_acc), p.E), p.Ntot, p.E, p.k,
                                            p.cap, p.ec ? 1 : 0, p.cfg.aux_alpha, stats);
  return cudaGetLastError();
}

cudaError_t launch_router(const Plan& p, const void* x, const moe_weights* w, int32_t* idx, float* gate,
                          float* logits, float* probs, void* stats, void* ws, cudaStream_t st,
                          int32_t* tile_counts, bool finalize) {
  RouterArgs a{};
  a.x = x;
  a.wr = w->w_router;
  a.logit_bias = w->logit_bias;
  a.logits_in = nullptr;
  a.idx = idx;
  a.gate = gate;
  a.logits = logits;
  a.probs = probs;
  a.acc = stats_acc_at(ws_at<uint8_t>(ws, p.stat_acc), p.E);
  a.tile_counts = tile_counts;
  a.status = status_ptr(p, ws);
  a.N = p.N;
  a.d = p.d;
  a.E = p.E;
  a.k = p.k;
  a.cap = p.cap;
  a.tile = p.tile;
  a.gating = p.cfg.gating;
  a.alpha = p.cfg.aux_alpha;
  cudaError_t err;
  if (router_uses_tc(p)) {
    // partial logits (K split) in the workspace, else the logits themselves
    const bool split = p.rsplit > 1;
    float* lg = logits ? logits : ws_at<float>(ws, p.L.logits);
    float* part = split ? ws_at<float>(ws, p.logits_part) : lg;
    err = launch_router_logits_tc(p, x, w->w_router, w->logit_bias, part, (int)p.rsplit, a.status, st);
    if (err != cudaSuccess) return err;
    a.logits_in = part;
    a.splits = p.rsplit;
    a.part_stride = p.N * p.E;
    a.logits = split ? logits : nullptr;  // unsplit: the GEMM wrote the logits (bias included)
    err = launch_router_logits_in<__nv_bfloat16>(p, a, st);
  } else if (router_uses_mma(p)) {
    err = (p.ec || p.k <= 2) ? launch_router_mma_k<2>(p, a, st) : launch_router_mma_k<8>(p, a, st);
  } else {
    err = p.bf16 ? launch_router_simt<__nv_bfloat16>(p, a, st) : launch_router_simt<float>(p, a, st);
  }
  if (err != cudaSuccess) return err;
  if (finalize) {
    router_finalize_kernel<<<1, 512, 0, st>>>(a.acc, p.Ntot, p.E, p.k, p.cap, p.ec ? 1 : 0, p.cfg.aux_alpha, stats);
  }
  return cudaGetLastError();
}

}  // namespace moe
