// Test kernel: runs the grouped GEMM epilogue's activation functions (the same
// device code, from the library's act.cuh) over arrays of inputs, so a test can
// compare them with the exact fp64 definitions over a dense sweep.
// which = 0: out[i] = GELU(a[i]); which = 1: out[i] = silu(a[i]) * b[i].
#include <cuda_runtime.h>

#include "act.cuh"

namespace {

__global__ void act_probe_kernel(int which, const float* a, const float* b, float* out, long long n_pairs) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_pairs) return;
  const float2 u = reinterpret_cast<const float2*>(a)[i];
  float2 r;
  if (which == 0) {
    r = moe::act::gelu2_as7128(u);
  } else {
    r = moe::act::silu_mul2(u, reinterpret_cast<const float2*>(b)[i]);
  }
  reinterpret_cast<float2*>(out)[i] = r;
}

}  // namespace

// a, b, out: device arrays of 2 * n_pairs floats (8-byte aligned); b unused for GELU.
extern "C" int act_probe(int which, const float* a, const float* b, float* out, long long n_pairs, void* stream) {
  if (n_pairs <= 0) return 0;
  const int threads = 256;
  const long long blocks = (n_pairs + threads - 1) / threads;
  act_probe_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(which, a, b, out, n_pairs);
  return (int)cudaGetLastError();
}
