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

// The same for more than 8 slices, with four lanes per group of 8 values
// (slices_to_bf16x8_4lanes; a site with at most 8 slices takes the one-thread tree). The four
// lanes of an item are consecutive threads of one warp, all active or all idle together.
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
    const int S = P.S;
    if (S <= 8) {   // a site of a grouped call with few slices: the one-thread tree
      if (l4 == 0) *reinterpret_cast<uint4*>(P.out + size_t(row) * R + g * 8) = slices_to_bf16x8(p, stride, S);
      continue;
    }
    const uint4 o = slices_to_bf16x8_4lanes(p, stride, S, l4, gmask);
    if (l4 == 0) *reinterpret_cast<uint4*>(P.out + size_t(row) * R + g * 8) = o;
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
