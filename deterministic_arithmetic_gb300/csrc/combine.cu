// combine.cu -- finishes the fixed summation tree of the weight gradients: the
// canonical tree over the chunk partials of every output (combine.cuh), one
// block per 128 outputs of every job.
#include "combine.cuh"

namespace lora {

__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ CombineJobs jobs) {
  grid_dependency_wait();
  grid_dependents_launch();
  combine_table_block(jobs, blockIdx.x);
}

cudaError_t launch_combine(const CombineJobs& jobs, cudaStream_t st) {
  if (jobs.n < 1 || jobs.n > 2 * kMaxSites) return cudaErrorInvalidValue;
  const int blocks = combine_table_blocks(jobs);
  if (blocks == 0) return cudaSuccess;
  return launch_pdl(combine_kernel, dim3(unsigned(blocks)), dim3(256), 0, st, jobs);
}

}  // namespace lora
