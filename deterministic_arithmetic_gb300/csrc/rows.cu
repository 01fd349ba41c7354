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
//
// The launch may also carry combine jobs (combine.cuh): in the backward pass,
// the dB tree over the chunk partials that the dy kernel has just written,
// while they are still in L2; those blocks follow the rows blocks.
#include <algorithm>

#include "combine.cuh"

namespace lora {

// FOUR: four lanes per item (some site has more than 8 slices; slices_to_bf16x8_4lanes),
// otherwise one thread per item. The first nrb blocks form rows; the rest run combine jobs.
template <bool GR, bool FOUR>
__global__ void __launch_bounds__(256)
    rows_kernel(const __grid_constant__ RowsArgs args, const __grid_constant__ CombineJobs cj, int nrb) {
  grid_dependency_wait();      // the partials of the preceding kernel are complete
  grid_dependents_launch();
  if (int(blockIdx.x) >= nrb) {
    combine_table_block(cj, int(blockIdx.x) - nrb);
    return;
  }
  const int R = args.R, RP = args.RP, G = R / 8;
  constexpr int L = FOUR ? 4 : 1;                     // lanes per item
  const int l4 = FOUR ? int(threadIdx.x & 3) : 0;
  const unsigned gmask = 0xFu << (threadIdx.x & 28u);
  // the L lanes of an item are consecutive threads of one warp, all active or all idle together
  for (int64_t i = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) / L; i < args.total;
       i += int64_t(nrb) * blockDim.x / L) {
    int k = 0;
    if constexpr (GR)
      while (k + 1 < args.n && i >= args.s[k + 1].item0) ++k;
    const RowsSite& P = args.s[k];
    const int64_t li = i - P.item0;
    const int64_t row = li / G;
    const int g = int(li % G);
    const float* p = P.part + size_t(row) * RP + g * 8;
    const size_t stride = size_t(P.M) * RP;
    uint4* out = reinterpret_cast<uint4*>(P.out + size_t(row) * R + g * 8);
    if (!FOUR || P.S <= 8) {   // the one-thread tree (in the four-lane form: lane 0 alone)
      if (l4 == 0) *out = slices_to_bf16x8(p, stride, P.S);
    } else {
      const uint4 o = slices_to_bf16x8_4lanes(p, stride, P.S, l4, gmask);
      if (l4 == 0) *out = o;
    }
  }
}

template <bool GR, bool FOUR>
static cudaError_t launch_inst(const RowsArgs& args, const CombineJobs& cj, int nrb, cudaStream_t st) {
  const int blocks = nrb + combine_table_blocks(cj);
  return launch_pdl(rows_kernel<GR, FOUR>, dim3(unsigned(blocks)), dim3(256), 0, st, args, cj, nrb);
}

cudaError_t launch_rows(RowsArgs& args, const CombineJobs* jobs, int nsm, cudaStream_t st) {
  if (args.n < 1 || args.n > kMaxSites) return cudaErrorInvalidValue;
  CombineJobs cj{};
  if (jobs) {
    if (jobs->n < 0 || jobs->n > 2 * kMaxSites) return cudaErrorInvalidValue;
    cj = *jobs;
  }
  int64_t item0 = 0;
  int smax = 0;
  for (int i = 0; i < args.n; ++i) {
    args.s[i].item0 = item0;
    item0 += int64_t(args.s[i].M) * (args.R / 8);
    smax = std::max(smax, args.s[i].S);
  }
  args.total = item0;
  const bool four = smax > 8;
  const int nrb = item0 == 0 ? 0 : int(std::min<int64_t>(ceil_div(item0 * (four ? 4 : 1), 256), int64_t(nsm) * 8));
  if (nrb + combine_table_blocks(cj) == 0) return cudaSuccess;
  if (four) return args.n > 1 ? launch_inst<true, true>(args, cj, nrb, st) : launch_inst<false, true>(args, cj, nrb, st);
  return args.n > 1 ? launch_inst<true, false>(args, cj, nrb, st) : launch_inst<false, false>(args, cj, nrb, st);
}

}  // namespace lora
