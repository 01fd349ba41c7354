// combine.cu -- finishes the fixed summation tree across work-unit partials.
//
// Every reduction of the operator is defined as: 16-term tensor-core leaves,
// added by the canonical pairwise tree over the leaf index. The down and
// weight-gradient kernels leave one FP32 partial per slice / row chunk (each a
// complete subtree over a power-of-two block of leaves); this kernel adds the
// S partials of each output element with the same canonical tree, in FP32,
// round to nearest, and writes the output: U and dU rounded to BF16 (the
// rounding points "round to BF16" / "D4" of page "[DSv4][P5-3]
// shared_grouped_lora_delta: CUDA + Triton, both batch-invariant", section
// "Summary"), dA and dB in FP32. No atomics: one thread owns one output.
#include <cuda_bf16.h>

#include <algorithm>

#include "kernels.h"

namespace lora {

// Canonical pairwise tree over p[0], p[stride], ..., p[(S-1)*stride]: after
// leaf i, merge once per trailing one bit of i; finally fold the remaining
// stack from the right. Equals the level-by-level tree where node i pairs
// with node i + 2^l whenever i is a multiple of 2^(l+1).
__device__ __forceinline__ float canonical_sum(const float* __restrict__ p, size_t stride, int S) {
  float stk[32];
  int top = 0;
  for (int i = 0; i < S; ++i) {
    float v = p[size_t(i) * stride];
    for (int t = i; t & 1; t >>= 1) v = __fadd_rn(stk[--top], v);
    stk[top++] = v;
  }
  if (top == 0) return 0.0f;
  float r = stk[--top];
  while (top > 0) r = __fadd_rn(stk[--top], r);
  return r;
}

__global__ void __launch_bounds__(256) combine_kernel(CombineJob j0, CombineJob j1) {
  const CombineJob& j = blockIdx.y == 0 ? j0 : j1;
  const size_t n = size_t(j.rows) * j.cols;
  for (size_t e = size_t(blockIdx.x) * blockDim.x + threadIdx.x; e < n; e += size_t(gridDim.x) * blockDim.x) {
    if (j.mode == 0) {            // part[S][rows][RP] -> bf16 out[rows][R]
      const size_t m = e / j.cols, r = e % j.cols;
      const float s = canonical_sum(j.part + m * j.RP + r, size_t(j.rows) * j.RP, j.S);
      reinterpret_cast<__nv_bfloat16*>(j.out)[e] = __float2bfloat16_rn(s);
    } else if (j.mode == 1) {     // part[S][RP][rows] -> fp32 out[rows][R]; threads run along rows
      const size_t r = e / j.rows, nidx = e % j.rows;
      const float s = canonical_sum(j.part + r * j.rows + nidx, size_t(j.RP) * j.rows, j.S);
      reinterpret_cast<float*>(j.out)[nidx * j.cols + r] = s;
    } else {                      // part[S][RP][cols] -> fp32 out[R][cols]
      const size_t r = e / j.cols, k = e % j.cols;
      const float s = canonical_sum(j.part + r * j.cols + k, size_t(j.RP) * j.cols, j.S);
      reinterpret_cast<float*>(j.out)[e] = s;
    }
  }
}

cudaError_t launch_combine(const CombineJob* jobs, int njobs, cudaStream_t st) {
  if (njobs < 1 || njobs > 2) return cudaErrorInvalidValue;
  size_t most = 0;
  for (int i = 0; i < njobs; ++i) most = std::max(most, size_t(jobs[i].rows) * jobs[i].cols);
  if (most == 0) return cudaSuccess;
  const unsigned bx = unsigned(std::min<size_t>((most + 255) / 256, 4096));
  combine_kernel<<<dim3(bx, njobs), 256, 0, st>>>(jobs[0], njobs > 1 ? jobs[1] : jobs[0]);
  return cudaGetLastError();
}

}  // namespace lora
