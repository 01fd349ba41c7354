// combine.cuh -- the canonical tree over the weight gradients' chunk partials, one block of
// 256 threads per 128 outputs (used by the combine kernel and, for dB, by the rows launch
// of the backward pass).
//
// Every reduction of the operator is defined as: 16-term tensor-core leaves,
// added by the canonical pairwise tree over the leaf index. The weight-gradient
// kernels leave one FP32 partial per 256-row chunk of the batch (each a
// complete subtree over a power-of-two block of leaves); a block adds the C
// chunk partials of each of its outputs with the canonical tree over the chunk
// index, in FP32, round to nearest ("dB = dV^T @ U", "dA = dU^T @ X" of page
// "[DSv4][P5-3] shared_grouped_lora_delta: CUDA + Triton, both
// batch-invariant", section "Summary"). No atomics: one block owns 128 outputs.
//
// A block = 8 warps x 32 lanes: lanes run along the contiguous output index,
// four outputs each (coalesced 16-byte reads of the [C][RP][cols] partials);
// warp w adds a contiguous power-of-two block of P chunks with all its loads
// in flight at once, and the eight warp results are added by a depth-3 tree.
// The whole is the canonical tree over the chunks (zero padding on the right
// changes no non-zero sum).
#pragma once

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

// Blocks of a job: one per 128 outputs of one row r of the [R][cols] view.
__host__ __device__ __forceinline__ int combine_blocks(const CombineJob& j) { return ((j.cols + 127) / 128) * j.R; }

// One block of a job: block index b in [0, combine_blocks(j)); every thread of the block calls this.
__device__ __forceinline__ void combine_block(const CombineJob& j, int b) {
  // chunks per warp: the smallest power of two with 8 * P >= C (warp blocks stay power-of-two aligned)
  int P = 1;
  while (8 * P < j.C) P *= 2;
  const int nx = (j.cols + 127) / 128;
  const int r = b / nx;
  const int col0 = (b % nx) * 128;
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
    const float4 c = add4(add4(wsum[4][lane], wsum[5][lane]), add4(wsum[6][lane], wsum[7][lane]));
    const float4 t = add4(a, c);
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

// Block b of a table of jobs (jobs in order, each combine_blocks(j) long).
__device__ __forceinline__ void combine_table_block(const CombineJobs& jobs, int b) {
  int k = 0;
  while (k + 1 < jobs.n && b >= combine_blocks(jobs.j[k])) b -= combine_blocks(jobs.j[k++]);
  combine_block(jobs.j[k], b);
}

inline int combine_table_blocks(const CombineJobs& jobs) {
  int t = 0;
  for (int i = 0; i < jobs.n; ++i) t += combine_blocks(jobs.j[i]);
  return t;
}

}  // namespace lora
