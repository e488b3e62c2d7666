// Internal launch interface of the library (host side). Not installed.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kRouterWarps = 8;
constexpr int kTileTokens = 32;  // permute tiles: one warp's 32 consecutive tokens

// Everything the launchers need, derived once from a validated moe_config.
struct Plan {
  moe_config cfg;
  int64_t N, d, F, E, S, Fs, k;
  bool bf16, swiglu, ec, bias;
  int64_t cap;       // C
  int64_t max_rows;  // rows reserved for xp / h / yp
  int64_t tiles;     // ceil(N / 32)
  int64_t words;     // ceil(E / 32): expert bitmap words per token (expert choice)
  int router_tpw;    // tokens per router warp
  int64_t router_blocks;
  moe_workspace_layout L;
  // scratch sub-buffers (byte offsets into the workspace)
  size_t part_p, part_cnt, part_lse;  // router partials
  size_t tile_counts, tile_base;      // permute [E][T], [E][T+1]
  size_t ec_bits;                     // [N][words]
  size_t logits_raw;                  // unused for now
};

moe_status make_plan(const moe_config* cfg, Plan* p);

inline int32_t* status_ptr(const Plan& p, void* ws) {
  return reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + p.L.status);
}
template <typename T>
inline T* ws_at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// router.cu
cudaError_t launch_router(const Plan& p, const void* x, const moe_weights* w, int32_t* idx, float* gate,
                          float* logits, float* probs, void* stats, void* ws, cudaStream_t st);

// permute.cu
cudaError_t launch_ec_select(const Plan& p, const float* probs, int32_t* idx, float* gate, void* ws,
                             cudaStream_t st);
cudaError_t launch_permute(const Plan& p, const void* x, const int32_t* idx, const float* gate, void* xp,
                           int32_t* tok_rows, int32_t* tok_off, int32_t* expert_off, int32_t* row_token,
                           float* row_gate, void* stats, void* ws, cudaStream_t st);
cudaError_t launch_combine(const Plan& p, const void* yp, const int32_t* tok_rows, const int32_t* tok_off,
                           const void* ys, void* out, cudaStream_t st);

// ffn_simt.cu (fp32 layers)
cudaError_t launch_ffn_f32(const Plan& p, const void* xp, const int32_t* expert_off, const float* row_gate,
                           const void* x, const moe_weights* w, void* h, void* hs, void* yp, void* ys,
                           int32_t* status, cudaStream_t st, int part);

// gemm_tc.cu (bf16 layers, tcgen05)
cudaError_t launch_ffn_bf16(const Plan& p, const void* xp, const int32_t* expert_off, const float* row_gate,
                            const void* x, const moe_weights* w, void* h, void* hs, void* yp, void* ys,
                            int32_t* status, cudaStream_t st, int part);
bool tc_gemm_available();

}  // namespace moe
