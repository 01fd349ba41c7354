// rows.cu -- the BF16 rows of U and dU from the slice partials:
//   U[m][r]  = bf16(canonical tree over the K-slices of the U partials)    ("U = X @ A^T", rounded)
//   dU[m][r] = bf16(canonical tree over the N-slices of the dU partials)   ("dU = dV @ B", rounded)
// (page "[DSv4][P5-3] shared_grouped_lora_delta: CUDA + Triton, both
// batch-invariant", section "Summary": FP32 accumulation, then one rounding to
// BF16 of the finished sum.)
//
// The down (or dy) kernel leaves one FP32 partial per (row, slice); each slice
// holds a power-of-two number of 16-term leaves, so the canonical tree over the
// slices finishes the canonical tree over all leaves. One thread forms 8
// consecutive values of one row: all its loads of a block of slices are in
// flight together, then it adds them in the tree's order and stores 16 bytes.
// Consecutive threads take consecutive 32-byte groups (coalesced reads and
// writes). The partials were just written by the preceding kernel and are read
// from L2 (cache-global loads). This is the only consumer of the partials, so
// every row is formed once; the up-projection that follows loads finished rows.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace lora {

template <bool GR>
__global__ void __launch_bounds__(256) rows_kernel(const __grid_constant__ RowsArgs args) {
  grid_dependency_wait();      // the partials of the preceding kernel are complete
  grid_dependents_launch();
  const int R = args.R, RP = args.RP, G = R / 8;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < args.total;
       i += int64_t(gridDim.x) * blockDim.x) {
    int k = 0;
    if constexpr (GR)
      while (k + 1 < args.n && i >= args.s[k + 1].item0) ++k;
    const RowsSite& P = args.s[k];
    const int64_t li = i - P.item0;
    const int64_t row = li / G;
    const int g = int(li % G);
    *reinterpret_cast<uint4*>(P.out + size_t(row) * R + g * 8) =
        slices_to_bf16x8(P.part + size_t(row) * RP + g * 8, size_t(P.M) * RP, P.S);
  }
}

// The same for more than 8 slices, with four lanes per group of 8 values: lane l adds block
// 4 s + l of 8 slices (every load of its block in flight; a partial last block is padded with
// zeros, as in the one-thread tree), the four block sums meet by shuffles in the canonical
// order (a block past the last one passes its partner up unchanged), and the sums of the
// 32-slice groups go through the canonical tree over the group index. Same bits as the
// one-thread tree of slices_to_bf16x8 for every slice count (a site with at most 8 slices
// takes that function itself: its zero padding differs, which decides the sign of a zero).
// The four lanes of an item are consecutive threads of one warp, all active or all idle
// together.
template <bool GR>
__global__ void __launch_bounds__(256) rows4_kernel(const __grid_constant__ RowsArgs args) {
  grid_dependency_wait();
  grid_dependents_launch();
  const int R = args.R, RP = args.RP, G = R / 8;
  const int l4 = threadIdx.x & 3;
  const unsigned gmask = 0xFu << (threadIdx.x & 28u);
  for (int64_t i = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 2; i < args.total;
       i += (int64_t(gridDim.x) * blockDim.x) >> 2) {
    int k = 0;
    if constexpr (GR)
      while (k + 1 < args.n && i >= args.s[k + 1].item0) ++k;
    const RowsSite& P = args.s[k];
    const int64_t li = i - P.item0;
    const int64_t row = li / G;
    const int g = int(li % G);
    const float* p = P.part + size_t(row) * RP + g * 8;
    const size_t stride = size_t(P.M) * RP;
    const int S = P.S, nb = (S + 7) / 8, nsg = (nb + 3) / 4;
    if (S <= 8) {   // a site of a grouped call with few slices: the one-thread tree
      if (l4 == 0) *reinterpret_cast<uint4*>(P.out + size_t(row) * R + g * 8) = slices_to_bf16x8(p, stride, S);
      continue;
    }
    float stk[24][8];
    int top = 0;
    for (int sg = 0; sg < nsg; ++sg) {
      const int b = 4 * sg + l4;
      float x[1][8];
      if (b < nb) {
        block_slices<8, 1>(p + size_t(b) * 8 * stride, stride, min(8, S - 8 * b), x);
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) x[0][c] = 0.0f;
      }
      // pairs (0, 1) and (2, 3): left + right, or left alone when the right block does not exist
      const bool has_right = 4 * sg + (l4 | 1) < nb;
      float pr[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float y = __shfl_xor_sync(gmask, x[0][c], 1, 4);
        const float left = (l4 & 1) ? y : x[0][c], right = (l4 & 1) ? x[0][c] : y;
        pr[c] = has_right ? __fadd_rn(left, right) : left;
      }
      // the two pairs: (0, 1) + (2, 3), or (0, 1) alone when block 2 does not exist
      const bool has_second = 4 * sg + 2 < nb;
      float sgs[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float y = __shfl_xor_sync(gmask, pr[c], 2, 4);
        const float first = (l4 & 2) ? y : pr[c], second = (l4 & 2) ? pr[c] : y;
        sgs[c] = has_second ? __fadd_rn(first, second) : first;
      }
      // canonical tree over the 32-slice groups: merge once per trailing one of sg
      for (int t = sg; t & 1; t >>= 1) {
        --top;
#pragma unroll
        for (int c = 0; c < 8; ++c) sgs[c] = __fadd_rn(stk[top][c], sgs[c]);
      }
#pragma unroll
      for (int c = 0; c < 8; ++c) stk[top][c] = sgs[c];
      ++top;
    }
    float o[8];
    --top;
#pragma unroll
    for (int c = 0; c < 8; ++c) o[c] = stk[top][c];
    while (top > 0) {
      --top;
#pragma unroll
      for (int c = 0; c < 8; ++c) o[c] = __fadd_rn(stk[top][c], o[c]);
    }
    if (l4 == 0) *reinterpret_cast<uint4*>(P.out + size_t(row) * R + g * 8) = pack_bf16x8(o);
  }
}

cudaError_t launch_rows(RowsArgs& args, int nsm, cudaStream_t st) {
  if (args.n < 1 || args.n > kMaxSites) return cudaErrorInvalidValue;
  int64_t item0 = 0;
  for (int i = 0; i < args.n; ++i) {
    args.s[i].item0 = item0;
    item0 += int64_t(args.s[i].M) * (args.R / 8);
  }
  args.total = item0;
  if (item0 == 0) return cudaSuccess;
  int smax = 0;
  for (int i = 0; i < args.n; ++i) smax = std::max(smax, args.s[i].S);
  if (smax > 8) {   // many slices: four lanes per item
    const int blocks = int(std::min<int64_t>(ceil_div(item0 * 4, 256), int64_t(nsm) * 8));
    if (args.n > 1) return launch_pdl(rows4_kernel<true>, dim3(blocks), dim3(256), 0, st, args);
    return launch_pdl(rows4_kernel<false>, dim3(blocks), dim3(256), 0, st, args);
  }
  const int blocks = int(std::min<int64_t>(ceil_div(item0, 256), int64_t(nsm) * 8));
  if (args.n > 1) return launch_pdl(rows_kernel<true>, dim3(blocks), dim3(256), 0, st, args);
  return launch_pdl(rows_kernel<false>, dim3(blocks), dim3(256), 0, st, args);
}

}  // namespace lora
