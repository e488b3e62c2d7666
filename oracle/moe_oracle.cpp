// moe_oracle.cpp -- TEST INFRASTRUCTURE, NOT PART OF THE LIBRARY.
//
// A plain, slow, single-threaded CPU definition of the forward pass of one
// top-k Mixture-of-Experts FFN layer, in fp64. Only the tests, the package's
// smoke check and the benchmark's CPU-baseline leg load it. It shares no code,
// header, table or constant with the CUDA library, and the CUDA library never
// loads it.
//
// Pages the definitions follow (cited by page title and section):
//  [AIG]  "Mixture of Experts" (aigrafen.se): the gate formula
//         y = sum_{i in top-k} g_i E_i(x), g = softmax(W_r x); the auxiliary
//         loss alpha * N * sum f_i P_i; the expert-capacity formula and the
//         dropping of tokens above it; the MoE module code (router without
//         bias, softmax, top-k, renormalisation of the chosen weights,
//         capacity int(cf*N*k/n), in-token-order truncation, GELU experts).
//  [AIE]  "Mixture of Experts (MoE)" (wiki.ai-engineering.at): router ->
//         softmax -> top-k -> weighted combination; top-k on scores then a
//         softmax over the k in its MoELayer code.
//  [VAN]  "MoE Architecture" (vanos001.github.io): router logits, top-k on
//         logits then softmax over the k; SwiGLUExpert and StandardExpert;
//         ExpertChoiceRouter; HybridMoE shared experts.
//  [STP]  "Mixture of Experts (MoE)" (learn.starphix.com): "Key Equations";
//         "Load Balancing (Critical)" (load_balancing_loss, z_loss);
//         "Shared + Specialized".
//
// Readings where the pages are silent or disagree are stated beside the code.
//
// Parity status: every function below is pinned by the CPU tests
// (tests/test_oracle_pins.py) against closed forms, invariants, brute force on
// tiny inputs, library routines and values the pages print, except where a
// comment says "parity unpinned".
//
// Build: g++ -O2 -shared -fPIC -o liboracle.so moe_oracle.cpp
// Defining ORACLE_PLANT=<n> compiles in one deliberate mistake (see the
// PLANT(...) sites); the tests use this to show that the pins catch it.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif
#define PLANT(n) (ORACLE_PLANT == (n))

extern "C" {

// Layer description. Field meaning is given in the oracle's Python wrapper.
struct OracleConfig {
  int64_t n_tokens, d_model, d_ff, n_experts, n_shared, d_ff_shared, top_k;
  double capacity_factor;  // <= 0: no capacity limit (token choice)
  int32_t gating;          // 0 softmax->top-k, 1 softmax->top-k->renormalise,
                           // 2 top-k on logits->softmax over k, 3 expert choice
  int32_t act;             // 0 GELU expert (Linear+bias, GELU, Linear+bias), 1 SwiGLU expert
  int32_t has_bias;        // biases present (GELU experts only)
  int32_t dtype;           // storage of x and all weights: 0 fp32, 1 bf16 bit patterns
  double aux_alpha;
  int32_t mimic_bf16;      // round the hidden activations and the final output to
                           // bf16, the two places a bf16 pipeline must store bf16
  int32_t passthrough;     // a token with no kept expert gets its input added (see
                           // oracle_combine_tokens)
  int32_t mx_act;          // routed experts compute in MXFP8: their input row and their
                           // hidden activations are quantised (oracle_mx_quantize)
                           // before each of their two matrix products
};

struct OracleWeights {
  const void* w_router;     // [E, d]
  const float* logit_bias;  // [E] or null
  const void* w1;           // [E, F, d]
  const void* w3;           // [E, F, d] (SwiGLU) or null
  const void* b1;           // [E, F] or null
  const void* w2;           // [E, d, F]
  const void* b2;           // [E, d] or null
  const void* ws1;          // [S, Fs, d]
  const void* ws3;          // [S, Fs, d] or null
  const void* bs1;          // [S, Fs] or null
  const void* ws2;          // [S, d, Fs]
  const void* bs2;          // [S, d] or null
};

}  // extern "C"

namespace {

// One stored element widened to double. bf16 is the upper half of an IEEE
// binary32, so widening is exact.
inline double load(const void* p, int64_t i, int32_t dtype) {
  if (dtype == 0) return static_cast<double>(static_cast<const float*>(p)[i]);
  uint32_t bits = static_cast<uint32_t>(static_cast<const uint16_t*>(p)[i]) << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return static_cast<double>(f);
}

// Round binary32 to the nearest bfloat16, ties to even (inputs are finite).
inline float round_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  u &= 0xFFFF0000u;
  float r;
  std::memcpy(&r, &u, sizeof r);
  return r;
}

inline double store_round(double v, const OracleConfig* c) {
  if (!c->mimic_bf16) return v;
  return static_cast<double>(round_bf16(static_cast<float>(v)));
}

// GELU as nn.GELU's default (exact erf form): 0.5 u (1 + erf(u / sqrt 2)).
// [AIG] MoE module code, [VAN] StandardExpert.
inline double gelu(double u) {
  if (PLANT(5)) return 0.5 * u * (1.0 + std::erf(u));
  return 0.5 * u * (1.0 + std::erf(u / std::sqrt(2.0)));
}

// ---------------------------------------------------------------------------
// FP8 E4M3 and the OCP microscaling (MX) block format "MXFP8". [STP] "Quantization"
// names lower-precision experts; the number formats are the Open Compute Project's:
// E4M3 is a sign bit, 4 exponent bits (bias 7) and 3 mantissa bits, exponent field 0
// subnormal (m/8 * 2^-6), largest finite magnitude 448 (1.75 * 2^8), no infinities;
// an MX block is 32 consecutive elements sharing one power-of-two scale 2^s whose
// E8M0 byte is s + 127.

// Nearest E4M3 magnitude to y >= 0, ties to the even code; anything above 448 gives
// 448 (saturating conversion). Returned as its code (7 bits, no sign).
inline uint8_t e4m3_code_sat(double y) {
  if (!(y < 448.0)) return 0x7E;  // 448
  int ex = 0;
  std::frexp(y, &ex);  // y = f * 2^ex, f in [0.5, 1): floor(log2 y) = ex - 1
  int E = ex - 1;
  if (y == 0.0 || E < -6) E = -6;  // subnormal range: the spacing of the lowest binade
  const double spacing = std::ldexp(1.0, E - 3);
  double r = std::nearbyint(y / spacing);  // round half to even (default rounding mode)
  if (PLANT(14)) r = std::floor(y / spacing + 0.5);  // ties away from zero
  int m = static_cast<int>(r);
  if (m >= 16) {  // rounded up into the next binade
    E += 1;
    m = 8;
  }
  if (m < 8) return static_cast<uint8_t>(m);  // subnormal (E == -6): code = m
  return static_cast<uint8_t>(((E + 7) << 3) | (m - 8));
}

inline double e4m3_code_value(uint8_t c) {
  const int e = (c >> 3) & 0xF, m = c & 7;
  const double mag = e == 0 ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
  return (c & 0x80) ? -mag : mag;
}

// One MX block of n <= 32 values: the shared exponent is s = floor(log2(max |v|)) - 8
// (8 = the exponent of E4M3's largest power of two, so the block maximum lands in
// [256, 512) before rounding and saturation), clamped to the E8M0 range [-127, 127];
// an all-zero block takes s = -127. Each element is the E4M3 code of v / 2^s.
inline void mx_block(const double* v, int n, uint8_t* codes, uint8_t* scale) {
  double amax = 0.0;
  for (int i = 0; i < n; ++i) amax = std::max(amax, std::fabs(v[i]));
  int s = -127;
  if (amax > 0.0) {
    int ex = 0;
    std::frexp(amax, &ex);
    s = (ex - 1) - (PLANT(13) ? 7 : 8);
    s = std::min(127, std::max(-127, s));
  }
  *scale = static_cast<uint8_t>(s + 127);
  for (int i = 0; i < n; ++i) {
    const uint8_t c = e4m3_code_sat(std::ldexp(std::fabs(v[i]), -s));
    codes[i] = std::signbit(v[i]) ? static_cast<uint8_t>(c | 0x80) : c;
  }
}

// v <- its MXFP8 value (quantise, then dequantise exactly), blocks of 32 along v.
inline void mx_round_trip(double* v, int64_t n) {
  uint8_t codes[32], scale;
  for (int64_t b = 0; b < n; b += 32) {
    const int m = static_cast<int>(std::min<int64_t>(32, n - b));
    mx_block(v + b, m, codes, &scale);
    for (int i = 0; i < m; ++i) v[b + i] = std::ldexp(e4m3_code_value(codes[i]), scale - 127);
  }
}

// SiLU: u * sigmoid(u). [VAN] SwiGLUExpert.
inline double silu(double u) {
  if (PLANT(6)) return u / (1.0 + std::exp(u));
  return u / (1.0 + std::exp(-u));
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// Expert capacity. [AIG] "Expert capacity": C = tokens / experts x capacity
// factor, and its MoE code int(cf * N * k / n); [VAN] CapacityManagedMoE uses
// the same N*k*cf/E. Reading: the layer takes C = ceil(N*k*cf/E) (the
// product is an exact integer on every workload here, where floor = ceil).
// cf <= 0 means no limit (C = N: an expert can hold at most every token once).
// Expert choice ([VAN] ExpertChoiceRouter: int(N*cf/E) tokens per expert)
// reads cf there as k*cf, so the same C = ceil(N*k*cf/E), capped at N.
int64_t oracle_capacity(const OracleConfig* c) {
  const int64_t N = c->n_tokens;
  if (c->capacity_factor <= 0.0) return N;
  double kk = static_cast<double>(c->top_k);
  if (PLANT(4)) kk = 1.0;
  double v = std::ceil(static_cast<double>(N) * kk * c->capacity_factor /
                       static_cast<double>(c->n_experts));
  int64_t cap = static_cast<int64_t>(v);
  if (cap > N) cap = N;
  if (cap < 0) cap = 0;
  return cap;
}

// ---------------------------------------------------------------------------
// Router linear: L[t,e] = sum_c x[t,c] W_r[e,c] (+ per-expert logit offset),
// accumulated in fp64 and rounded once to fp32. [STP] "Key Equations":
// router_logits = x @ W_router^T; [AIG] nn.Linear(d, n, bias=False).
void oracle_router_logits(const OracleConfig* c, const void* x, const OracleWeights* w,
                          float* logits) {
  const int64_t N = c->n_tokens, d = c->d_model, E = c->n_experts;
  for (int64_t t = 0; t < N; ++t) {
    for (int64_t e = 0; e < E; ++e) {
      double s = 0.0;
      for (int64_t i = 0; i < d; ++i)
        s += load(x, t * d + i, c->dtype) * load(w->w_router, e * d + i, c->dtype);
      if (w->logit_bias) s += static_cast<double>(w->logit_bias[e]);
      logits[t * E + e] = static_cast<float>(s);
    }
  }
}

// ---------------------------------------------------------------------------
// Softmax over experts and its log-normaliser, in fp64.
// p[t,e] = exp(L[t,e] - lse_t), lse_t = m + log sum_e exp(L[t,e] - m), m = max_e L.
// [AIG] g = softmax(W_r x); [STP] z_loss uses logsumexp of the router logits.
void oracle_softmax(int64_t N, int64_t E, const float* logits, double* probs, double* lse) {
  for (int64_t t = 0; t < N; ++t) {
    const float* L = logits + t * E;
    double m = L[0];
    for (int64_t e = 1; e < E; ++e) m = std::max(m, static_cast<double>(L[e]));
    double s = 0.0;
    for (int64_t e = 0; e < E; ++e) s += std::exp(static_cast<double>(L[e]) - m);
    double l = m + std::log(s);
    lse[t] = l;
    for (int64_t e = 0; e < E; ++e) probs[t * E + e] = std::exp(static_cast<double>(L[e]) - l);
  }
}

// ---------------------------------------------------------------------------
// Top-k experts per token, by logit, descending; equal logits go to the lower
// expert index. Reading: [AIG]/[AIE] take top-k on the softmax probabilities,
// [VAN]/[STP] on the logits; softmax is strictly increasing, so both select
// the same set, and ranking the fp32 logits avoids ties created by rounding
// of exp. Plain repeated arg-max.
void oracle_topk(int64_t N, int64_t E, int64_t k, const float* logits, int32_t* idx) {
  std::vector<char> taken(static_cast<size_t>(E));
  for (int64_t t = 0; t < N; ++t) {
    const float* L = logits + t * E;
    std::fill(taken.begin(), taken.end(), 0);
    for (int64_t j = 0; j < k; ++j) {
      int64_t best = -1;
      for (int64_t e = 0; e < E; ++e) {
        if (taken[e]) continue;
        bool better = best < 0 || L[e] > L[best];
        if (PLANT(2)) better = best < 0 || L[e] >= L[best];
        if (better) best = e;
      }
      taken[best] = 1;
      idx[t * k + j] = static_cast<int32_t>(best);
    }
  }
}

// ---------------------------------------------------------------------------
// Gate values of the chosen experts, in fp64.
//  gating 0: g_j = p[t, idx_j]                ([AIG] formula; [AIE] "Gate: Softmax")
//  gating 1: g_j = p_j / sum_j' p_j'          ([AIG] MoE code, "normalise the chosen ones")
//  gating 2: g_j = softmax over the k logits  ([VAN] TokenChoiceRouter, [STP] TopKRouter, [AIE] MoELayer)
void oracle_gates(const OracleConfig* c, const float* logits, const int32_t* idx, double* gate) {
  const int64_t N = c->n_tokens, E = c->n_experts, k = c->top_k;
  std::vector<double> p(static_cast<size_t>(E)), lse(1);
  for (int64_t t = 0; t < N; ++t) {
    const float* L = logits + t * E;
    const int32_t* I = idx + t * k;
    double* g = gate + t * k;
    if (c->gating == 2) {
      double m = L[I[0]];
      for (int64_t j = 1; j < k; ++j) m = std::max(m, static_cast<double>(L[I[j]]));
      double s = 0.0;
      for (int64_t j = 0; j < k; ++j) s += std::exp(static_cast<double>(L[I[j]]) - m);
      for (int64_t j = 0; j < k; ++j) g[j] = std::exp(static_cast<double>(L[I[j]]) - m) / s;
      continue;
    }
    oracle_softmax(1, E, L, p.data(), lse.data());
    double s = 0.0;
    for (int64_t j = 0; j < k; ++j) s += p[I[j]];
    for (int64_t j = 0; j < k; ++j) {
      g[j] = p[I[j]];
      if (c->gating == 1 && !PLANT(7)) g[j] /= s;
    }
  }
}

// ---------------------------------------------------------------------------
// Capacity and in-token-order dropping (token choice). For each expert the
// assignments (t, j) are ranked in ascending token order; rank < C is kept,
// the rest dropped. [AIG] MoE code: nonzero() of the expert's mask lists tokens
// in index order and index[:capacity] keeps the first C; [AIG] "Tokens above
// the limit are dropped". A token's k experts are distinct, so the order is
// total. Kept rows are numbered expert by expert (expert_off = exclusive
// prefix of kept counts), in token order within an expert.
//  row_of[t*k+j]  = row of (t, j), or -1 if dropped
//  expert_off[E+1], counts[E] (before dropping), kept[E]; returns the number dropped.
int64_t oracle_assign(const OracleConfig* c, const int32_t* idx, int64_t cap, int32_t* row_of,
                      int32_t* expert_off, int32_t* counts, int32_t* kept) {
  const int64_t N = c->n_tokens, E = c->n_experts, k = c->top_k;
  std::vector<int64_t> rank(static_cast<size_t>(N * k));
  for (int64_t e = 0; e < E; ++e) counts[e] = 0;
  if (PLANT(8)) {
    for (int64_t t = N - 1; t >= 0; --t)
      for (int64_t j = 0; j < k; ++j) rank[t * k + j] = counts[idx[t * k + j]]++;
  } else {
    for (int64_t t = 0; t < N; ++t)
      for (int64_t j = 0; j < k; ++j) rank[t * k + j] = counts[idx[t * k + j]]++;
  }
  int64_t dropped = 0;
  expert_off[0] = 0;
  for (int64_t e = 0; e < E; ++e) {
    kept[e] = static_cast<int32_t>(std::min<int64_t>(counts[e], cap));
    dropped += counts[e] - kept[e];
    expert_off[e + 1] = expert_off[e] + kept[e];
  }
  for (int64_t t = 0; t < N; ++t)
    for (int64_t j = 0; j < k; ++j) {
      int32_t e = idx[t * k + j];
      int64_t r = rank[t * k + j];
      row_of[t * k + j] = r < cap ? static_cast<int32_t>(expert_off[e] + r) : -1;
    }
  return dropped;
}

// ---------------------------------------------------------------------------
// The same capacity rule for one contiguous shard of a batch's tokens: base[e]
// assignments to expert e come from the tokens before the shard, so the shard's
// (t, j) has rank base[e] + (its rank among the shard's assignments to e) in the
// whole batch's token order, and is kept when that rank is below C. Rows number
// the shard's kept pairs expert by expert, in token order within an expert.
// [AIG] "Expert capacity" and MoE code (nonzero()[:capacity] over the batch).
// With base = 0 this is oracle_assign. Returns the shard's dropped count.
int64_t oracle_assign_shard(const OracleConfig* c, const int32_t* idx, int64_t cap, const int32_t* base,
                            int32_t* row_of, int32_t* expert_off, int32_t* counts, int32_t* kept) {
  const int64_t N = c->n_tokens, E = c->n_experts, k = c->top_k;
  std::vector<int64_t> rank(static_cast<size_t>(N * k));
  for (int64_t e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t t = 0; t < N; ++t)
    for (int64_t j = 0; j < k; ++j) rank[t * k + j] = counts[idx[t * k + j]]++;
  int64_t dropped = 0;
  expert_off[0] = 0;
  for (int64_t e = 0; e < E; ++e) {
    const int64_t left = std::max<int64_t>(cap - base[e], 0);
    kept[e] = static_cast<int32_t>(std::min<int64_t>(counts[e], left));
    dropped += counts[e] - kept[e];
    expert_off[e + 1] = expert_off[e] + kept[e];
  }
  for (int64_t t = 0; t < N; ++t)
    for (int64_t j = 0; j < k; ++j) {
      int32_t e = idx[t * k + j];
      int64_t r = rank[t * k + j];
      const int64_t global_rank = PLANT(12) ? r : base[e] + r;
      row_of[t * k + j] = global_rank < cap ? static_cast<int32_t>(expert_off[e] + r) : -1;
    }
  return dropped;
}

// ---------------------------------------------------------------------------
// Expert choice: every expert takes the C tokens with the largest key
// (its softmax-over-experts probability), ties to the lower token index, and
// lists them in ascending token order. [VAN] ExpertChoiceRouter (each expert
// takes topk(capacity) tokens); [AIG] "expert choice instead of token choice".
// Reading: [VAN]'s snippet takes the softmax over tokens (dim=0); this layer
// ranks by the softmax over experts, the same probability the gates use
// everywhere else on the pages. sel[e*C + c] = token id.
void oracle_expert_choice(const OracleConfig* c, const float* keys, int64_t cap, int32_t* sel) {
  const int64_t N = c->n_tokens, E = c->n_experts;
  std::vector<int32_t> order(static_cast<size_t>(N));
  for (int64_t e = 0; e < E; ++e) {
    for (int64_t t = 0; t < N; ++t) order[t] = static_cast<int32_t>(t);
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
      return keys[a * E + e] > keys[b * E + e];
    });
    std::vector<int32_t> chosen(order.begin(), order.begin() + cap);
    std::sort(chosen.begin(), chosen.end());
    for (int64_t i = 0; i < cap; ++i) sel[e * cap + i] = chosen[i];
  }
}

// ---------------------------------------------------------------------------
// Balancing statistics, in fp64.
//  f_e = (assignments routed to e before dropping) / (all assignments)
//  P_e = mean_t p[t,e]
//  aux = alpha * E * sum_e f_e P_e       ([AIG] "L_aux = alpha * N * sum f_i P_i",
//                                          N there being the number of experts)
//  z   = (mean_t lse_t)^2                ([STP] z_loss: logsumexp(...).mean() ** 2)
//  mean_lse_sq = mean_t lse_t^2          (the other common reading of "z-loss")
// Reading: f as the share of the N*k assignments ([STP] load_balancing_loss
// takes the mean of the one-hot top-k mask), so sum_e f_e = 1 and the loss is
// alpha at a uniform distribution; [AIG]'s code counts tokens (sum f = k) and
// drops alpha, both rejected. counts[E] are the per-expert assignment counts
// (token choice: before dropping; expert choice: C each).
// out[0] = aux, out[1] = z, out[2] = mean_lse_sq.
void oracle_stats(const OracleConfig* c, const float* logits, const int32_t* counts, double* f,
                  double* P, double* out) {
  const int64_t N = c->n_tokens, E = c->n_experts;
  std::vector<double> p(static_cast<size_t>(E)), lse(1);
  for (int64_t e = 0; e < E; ++e) P[e] = 0.0;
  double s_lse = 0.0, s_lse2 = 0.0;
  for (int64_t t = 0; t < N; ++t) {
    oracle_softmax(1, E, logits + t * E, p.data(), lse.data());
    for (int64_t e = 0; e < E; ++e) P[e] += p[e];
    s_lse += lse[0];
    s_lse2 += lse[0] * lse[0];
  }
  double total = 0.0;
  for (int64_t e = 0; e < E; ++e) total += counts[e];
  double aux = 0.0;
  for (int64_t e = 0; e < E; ++e) {
    P[e] /= static_cast<double>(N);
    f[e] = total > 0 ? counts[e] / total : 0.0;
    aux += f[e] * P[e];
  }
  double scale = PLANT(9) ? c->aux_alpha : c->aux_alpha * static_cast<double>(E);
  out[0] = scale * aux;
  double ml = s_lse / static_cast<double>(N);
  out[1] = PLANT(10) ? ml : ml * ml;
  out[2] = s_lse2 / static_cast<double>(N);
}

// ---------------------------------------------------------------------------
// One expert applied to one token, in fp64.
//  GELU expert   ([AIG] nn.Sequential(Linear(d,h), GELU(), Linear(h,d)); [VAN] StandardExpert):
//      h = gelu(W1 x + b1), y = W2 h + b2      (dropout is the identity at inference)
//  SwiGLU expert ([VAN] SwiGLUExpert; [STP] Expert, whose gate/w1 names are swapped):
//      h = silu(W1 x) * (W3 x), y = W2 h
// W1/W3 are [F, d] and W2 is [d, F] (nn.Linear [out, in]). shared != 0 selects
// the always-on shared expert e instead of routed expert e.
void oracle_expert_apply(const OracleConfig* c, const OracleWeights* w, int32_t shared, int64_t e,
                         const double* x, double* y) {
  const int64_t d = c->d_model;
  const int64_t F = shared ? c->d_ff_shared : c->d_ff;
  const void* W1 = shared ? w->ws1 : w->w1;
  const void* W3 = shared ? w->ws3 : w->w3;
  const void* B1 = shared ? w->bs1 : w->b1;
  const void* W2 = shared ? w->ws2 : w->w2;
  const void* B2 = shared ? w->bs2 : w->b2;
  const int32_t dt = c->dtype;
  // MXFP8 routed experts: the input row and (below) the hidden row are quantised
  const bool mx = c->mx_act && !shared;
  std::vector<double> xq(x, x + d);
  if (mx) mx_round_trip(xq.data(), d);
  x = xq.data();
  std::vector<double> h(static_cast<size_t>(F));
  for (int64_t f = 0; f < F; ++f) {
    double a = 0.0;
    for (int64_t i = 0; i < d; ++i) a += load(W1, (e * F + f) * d + i, dt) * x[i];
    if (c->act == 0) {
      if (c->has_bias && !PLANT(1)) a += load(B1, e * F + f, dt);
      h[f] = gelu(a);
    } else {
      double b = 0.0;
      for (int64_t i = 0; i < d; ++i) b += load(W3, (e * F + f) * d + i, dt) * x[i];
      h[f] = silu(a) * b;
    }
    if (!mx) h[f] = store_round(h[f], c);
  }
  if (mx && !PLANT(15)) mx_round_trip(h.data(), F);
  for (int64_t n = 0; n < d; ++n) {
    double s = 0.0;
    for (int64_t f = 0; f < F; ++f) {
      int64_t wi = PLANT(3) ? (e * F + f) * d + n : (e * d + n) * F + f;
      s += load(W2, wi, dt) * h[f];
    }
    if (c->act == 0 && c->has_bias) s += load(B2, e * d + n, dt);
    y[n] = s;
  }
}

// ---------------------------------------------------------------------------
// Layer output for the listed tokens, given the routing.
//  token choice: out[t] = sum_s shared_s(x_t) + sum_{j kept} g_{t,j} E_{idx_{t,j}}(x_t)
//  expert choice: out[t] = sum_s shared_s(x_t) + sum_{e : t in sel_e, ascending e} p[t,e] E_e(x_t)
// [AIG] y = sum g_i E_i(x) and its MoE code (out[index] += w * expert(x));
// [VAN] HybridMoE and [STP] SharedExpertMoE add the shared experts with weight 1.
// A dropped slot adds nothing ([AIG]: dropped tokens pass through the residual,
// which is outside this layer). With passthrough set, a token left with no kept
// expert (all its slots dropped; in expert choice, picked by no expert) adds its
// own input after the shared experts: [VAN] CapacityManagedMoE, "Handle dropped
// tokens (pass through residual)". Token-choice inputs: idx/gate [N,k], row_of
// [N,k] (-1 = dropped). Expert-choice inputs: sel [E,C], gate_ec [E,C].
void oracle_combine_tokens(const OracleConfig* c, const void* x, const OracleWeights* w,
                           const int32_t* idx, const double* gate, const int32_t* row_of,
                           const int32_t* sel, const double* gate_ec, int64_t cap,
                           const int64_t* tokens, int64_t n_out, double* out) {
  const int64_t d = c->d_model, k = c->top_k, E = c->n_experts;
  std::vector<double> xr(static_cast<size_t>(d)), y(static_cast<size_t>(d)),
      acc(static_cast<size_t>(d)), sh(static_cast<size_t>(d));
  for (int64_t o = 0; o < n_out; ++o) {
    const int64_t t = tokens[o];
    for (int64_t i = 0; i < d; ++i) xr[i] = load(x, t * d + i, c->dtype);
    std::fill(sh.begin(), sh.end(), 0.0);
    for (int64_t s = 0; s < c->n_shared; ++s) {
      oracle_expert_apply(c, w, 1, s, xr.data(), y.data());
      for (int64_t i = 0; i < d; ++i) sh[i] += y[i];
    }
    for (int64_t i = 0; i < d; ++i) acc[i] = sh[i];
    int64_t terms = 0;
    auto add_term = [&](int64_t e, double g) {
      oracle_expert_apply(c, w, 0, e, xr.data(), y.data());
      for (int64_t i = 0; i < d; ++i) acc[i] += g * y[i];
      ++terms;
    };
    if (c->gating == 3) {
      for (int64_t e = 0; e < E; ++e)
        for (int64_t i = 0; i < cap; ++i)
          if (sel[e * cap + i] == t) add_term(e, gate_ec[e * cap + i]);
    } else {
      for (int64_t j = 0; j < k; ++j)
        if (row_of[t * k + j] >= 0) add_term(idx[t * k + j], gate[t * k + j]);
    }
    bool pass = c->passthrough && terms == 0;
    if (PLANT(11) && c->passthrough && c->gating != 3) {  // any dropped slot passes the token through
      pass = false;
      for (int64_t j = 0; j < k; ++j) pass = pass || row_of[t * k + j] < 0;
    }
    if (pass)
      for (int64_t i = 0; i < d; ++i) acc[i] += xr[i];
    for (int64_t i = 0; i < d; ++i) out[o * d + i] = store_round(acc[i], c);
  }
}

// The bf16 rounding the mimic mode applies (exported for its pin): nearest, ties to even.
float oracle_round_bf16(float v) { return round_bf16(v); }

// MXFP8 quantisation of n values (n % 32 == 0): E4M3 codes [n] and E8M0 scale bytes
// [n / 32], the rule mx_block states (exported for its pins and the code-level checks).
void oracle_mx_quantize(const double* v, int64_t n, uint8_t* codes, uint8_t* scales) {
  for (int64_t b = 0; b < n; b += 32) mx_block(v + b, 32, codes + b, scales + b / 32);
}

// Routing entropy of a usage distribution, -sum p ln p over p > 0.
// [AIG] collapse detector ("Logging the routing entropy").
double oracle_entropy(const double* p, int64_t n) {
  double h = 0.0;
  for (int64_t i = 0; i < n; ++i)
    if (p[i] > 0) h -= p[i] * std::log(p[i]);
  return h;
}

}  // extern "C"
