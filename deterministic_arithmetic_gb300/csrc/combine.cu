// combine.cu -- finishes the fixed summation tree of the weight gradients.
//
// Every reduction of the operator is defined as: 16-term tensor-core leaves,
// added by the canonical pairwise tree over the leaf index. The weight-gradient
// kernels leave one FP32 partial per 256-row chunk of the batch (each a
// complete subtree over a power-of-two block of leaves); this kernel adds the
// C chunk partials of each element of dA and dB with the canonical tree over
// the chunk index, in FP32, round to nearest ("dB = dV^T @ U", "dA = dU^T @ X"
// of page "[DSv4][P5-3] shared_grouped_lora_delta: CUDA + Triton, both
// batch-invariant", section "Summary"). No atomics: one block owns 128 outputs.
//
// A block = 8 warps x 32 lanes: lanes run along the contiguous output index,
// four outputs each (coalesced 16-byte reads of the [C][RP][cols] partials);
// warp w adds a contiguous power-of-two block of P chunks with all its loads
// in flight at once, and the eight warp results are added by a depth-3 tree.
// The whole is the canonical tree over the chunks (zero padding on the right
// changes no non-zero sum).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace lora {

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
}

// canonical tree over n <= 8 float4 values p[0], p[stride], ... (zero padded to 8)
__device__ __forceinline__ float4 tree8_strided4(const float* __restrict__ p, size_t stride, int n) {
  float4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    v[i] = i < n ? __ldcg(reinterpret_cast<const float4*>(p + size_t(i) * stride)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int w = 1; w < 8; w <<= 1)
#pragma unroll
    for (int i = 0; i < 8; i += 2 * w) v[i] = add4(v[i], v[i + w]);
  return v[0];
}

// canonical tree over n float4 values (any n >= 1): blocks of 8, then the canonical tree over blocks
__device__ __forceinline__ float4 canonical_strided4(const float* __restrict__ p, size_t stride, int n) {
  if (n <= 8) return tree8_strided4(p, stride, n);
  float4 stk[32];
  int top = 0;
  for (int b = 0; b * 8 < n; ++b) {
    float4 x = tree8_strided4(p + size_t(b) * 8 * stride, stride, min(8, n - 8 * b));
    for (int t = b; t & 1; t >>= 1) x = add4(stk[--top], x);
    stk[top++] = x;
  }
  float4 r = stk[--top];
  while (top > 0) r = add4(stk[--top], r);
  return r;
}

__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ CombineJobs jobs) {
  grid_dependency_wait();
  grid_dependents_launch();
  const CombineJob& j = jobs.j[blockIdx.z];
  // chunks per warp: the smallest power of two with 8 * P >= C (warp blocks stay power-of-two aligned)
  int P = 1;
  while (8 * P < j.C) P *= 2;
  const int r = blockIdx.y;
  const int col0 = blockIdx.x * 128;
  if (r >= j.R || col0 >= j.cols) return;                // uniform over the block
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col = col0 + 4 * lane;                       // cols is a multiple of 8: all four in or all out
  __shared__ float4 wsum[8][32];
  const int c0 = warp * P;
  const int n = max(0, min(P, j.C - c0));
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  if (col < j.cols && n > 0) {
    const size_t stride = size_t(j.RP) * j.cols;
    s = canonical_strided4(j.part + size_t(c0) * stride + size_t(r) * j.cols + col, stride, n);
  }
  wsum[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && col < j.cols) {
    const float4 a = add4(add4(wsum[0][lane], wsum[1][lane]), add4(wsum[2][lane], wsum[3][lane]));
    const float4 b = add4(add4(wsum[4][lane], wsum[5][lane]), add4(wsum[6][lane], wsum[7][lane]));
    const float4 t = add4(a, b);
    if (j.transpose) {
      j.out[size_t(col) * j.R + r] = t.x;
      j.out[size_t(col + 1) * j.R + r] = t.y;
      j.out[size_t(col + 2) * j.R + r] = t.z;
      j.out[size_t(col + 3) * j.R + r] = t.w;
    } else {
      *reinterpret_cast<float4*>(j.out + size_t(r) * j.cols + col) = t;
    }
  }
}

cudaError_t launch_combine(const CombineJobs& jobs, cudaStream_t st) {
  if (jobs.n < 1 || jobs.n > 2 * kMaxSites) return cudaErrorInvalidValue;
  int cmax = 0, colmax = 0, rmax = 0;
  for (int i = 0; i < jobs.n; ++i) {
    cmax = std::max(cmax, jobs.j[i].C);
    colmax = std::max(colmax, jobs.j[i].cols);
    rmax = std::max(rmax, jobs.j[i].R);
  }
  if (cmax == 0 || colmax == 0) return cudaSuccess;
  const dim3 grid(unsigned((colmax + 127) / 128), unsigned(rmax), unsigned(jobs.n));
  return launch_pdl(combine_kernel, grid, dim3(256), 0, st, jobs);
}

}  // namespace lora
