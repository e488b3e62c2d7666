// Expert FFNs for fp32 layers, in fp32 FMA on the CUDA cores (tf32 tensor
// cores would not meet a 1e-4 relative tolerance). One thread per output
// element; the expert of a permuted row is found by binary search in
// expert_off. These layers are tiny (the fp32 workload is 64 tokens), so the
// kernels are written for clarity, not speed.
//
// Pages: "MoE Architecture" (vanos001.github.io) StandardExpert
// (w2(gelu(w1 x)), nn.Linear with bias) and SwiGLUExpert (w2(silu(w1 x) * w3 x));
// "Mixture of Experts" (aigrafen.se) MoE experts Linear -> GELU -> Linear;
// HybridMoE / "Shared + Specialized": shared experts on every token, weight 1.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

__device__ __forceinline__ int group_of_row(const int32_t* off, int64_t E, int64_t r) {
  int64_t lo = 0, hi = E;  // last e with off[e] <= r
  while (hi - lo > 1) {
    const int64_t mid = (lo + hi) >> 1;
    if (off[mid] <= r) lo = mid; else hi = mid;
  }
  return (int)lo;
}

__device__ __forceinline__ float gelu_erf(float u) { return 0.5f * u * (1.f + erff(u * 0.70710678118654752f)); }
__device__ __forceinline__ float silu(float u) { return u / (1.f + expf(-u)); }

// H[r, g*col_per_group + f] = act(A[r] . W1[g, f] (+ B1[g, f])) (SwiGLU: silu(A W1) * (A W3))
__global__ void up_f32_kernel(const float* __restrict__ A, int64_t rows, const int32_t* __restrict__ off,
                              int64_t E, const float* __restrict__ W1, const float* __restrict__ W3,
                              const float* __restrict__ B1, int64_t F, int64_t d, int swiglu,
                              float* __restrict__ H, int64_t ldh, int64_t col_per_group) {
  const int64_t f = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t r = (int64_t)blockIdx.y * blockDim.y + threadIdx.y;
  if (f >= F) return;
  int g;
  if (off) {
    if (r >= off[E]) return;
    g = group_of_row(off, E, r);
  } else {
    if (r >= rows) return;
    g = blockIdx.z;
  }
  const float* a = A + r * d;
  const float* w1 = W1 + ((int64_t)g * F + f) * d;
  float s1 = 0.f;
  for (int64_t i = 0; i < d; ++i) s1 = fmaf(a[i], w1[i], s1);
  float h;
  if (swiglu) {
    const float* w3 = W3 + ((int64_t)g * F + f) * d;
    float s3 = 0.f;
    for (int64_t i = 0; i < d; ++i) s3 = fmaf(a[i], w3[i], s3);
    h = silu(s1) * s3;
  } else {
    if (B1) s1 += B1[(int64_t)g * F + f];
    h = gelu_erf(s1);
  }
  H[r * ldh + (int64_t)g * col_per_group + f] = h;
}

// routed: Y[r, n] = gate[r] * (H[r] . W2[g, n] + B2[g, n])
// shared: Y[t, n] = sum_s (Hs[t, s*F:(s+1)*F] . Ws2[s, n] + Bs2[s, n])
__global__ void down_f32_kernel(const float* __restrict__ H, int64_t rows, const int32_t* __restrict__ off,
                                int64_t G, const float* __restrict__ W2, const float* __restrict__ B2,
                                const float* __restrict__ gate, int64_t F, int64_t d, float* __restrict__ Y) {
  const int64_t n = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t r = (int64_t)blockIdx.y * blockDim.y + threadIdx.y;
  if (n >= d) return;
  if (off) {
    if (r >= off[G]) return;
    const int g = group_of_row(off, G, r);
    const float* h = H + r * F;
    const float* w = W2 + ((int64_t)g * d + n) * F;
    float s = 0.f;
    for (int64_t f = 0; f < F; ++f) s = fmaf(h[f], w[f], s);
    if (B2) s += B2[(int64_t)g * d + n];
    Y[r * d + n] = gate[r] * s;
  } else {
    if (r >= rows) return;
    float s = 0.f;
    for (int64_t g = 0; g < G; ++g) {
      const float* h = H + r * (G * F) + g * F;
      const float* w = W2 + (g * d + n) * F;
      float sg = 0.f;
      for (int64_t f = 0; f < F; ++f) sg = fmaf(h[f], w[f], sg);
      if (B2) sg += B2[g * d + n];
      s += sg;
    }
    Y[r * d + n] = s;
  }
}

}  // namespace

// part: bit 0 = up-projections, bit 1 = down-projections.
cudaError_t launch_ffn_f32(const Plan& p, const void* xp, const int32_t* expert_off, const float* row_gate,
                           const void* x, const moe_weights* w, void* h, void* hs, void* yp, void* ys,
                           int32_t* status, cudaStream_t st, int part) {
  (void)status;
  const dim3 blk(32, 8);
  if (part & 1) {
    dim3 g1((unsigned)ceil_div(p.F, 32), (unsigned)ceil_div(p.max_rows, 8), 1);
    up_f32_kernel<<<g1, blk, 0, st>>>(static_cast<const float*>(xp), p.max_rows, expert_off, p.E,
                                      static_cast<const float*>(w->w1), static_cast<const float*>(w->w3),
                                      static_cast<const float*>(w->b1), p.F, p.d, p.swiglu ? 1 : 0,
                                      static_cast<float*>(h), p.F, 0);
    if (p.S > 0) {
      dim3 g2((unsigned)ceil_div(p.Fs, 32), (unsigned)ceil_div(p.N, 8), (unsigned)p.S);
      up_f32_kernel<<<g2, blk, 0, st>>>(static_cast<const float*>(x), p.N, nullptr, p.S,
                                        static_cast<const float*>(w->ws1), static_cast<const float*>(w->ws3),
                                        static_cast<const float*>(w->bs1), p.Fs, p.d, p.swiglu ? 1 : 0,
                                        static_cast<float*>(hs), p.S * p.Fs, p.Fs);
    }
  }
  if (part & 2) {
    dim3 g3((unsigned)ceil_div(p.d, 32), (unsigned)ceil_div(p.max_rows, 8), 1);
    down_f32_kernel<<<g3, blk, 0, st>>>(static_cast<const float*>(h), p.max_rows, expert_off, p.E,
                                        static_cast<const float*>(w->w2), static_cast<const float*>(w->b2), row_gate,
                                        p.F, p.d, static_cast<float*>(yp));
    if (p.S > 0) {
      dim3 g4((unsigned)ceil_div(p.d, 32), (unsigned)ceil_div(p.N, 8), 1);
      down_f32_kernel<<<g4, blk, 0, st>>>(static_cast<const float*>(hs), p.N, nullptr, p.S,
                                          static_cast<const float*>(w->ws2), static_cast<const float*>(w->bs2),
                                          nullptr, p.Fs, p.d, static_cast<float*>(ys));
    }
  }
  return cudaGetLastError();
}

}  // namespace moe
