// dvf32.cu -- the FP32-dY input of the backward pass: dV = bf16(fp32(dY * alpha))
// with dY read as binary32 (one FP32 multiply, round to nearest, then round to
// nearest even to BF16: the two rounding points of dV in page "[DSv4][P5-3]
// shared_grouped_lora_delta: CUDA + Triton, both batch-invariant", section
// "Summary", "D4"). The BF16 dV is written once to the workspace; the backward
// kernels then read it as their dY with alpha = 1, which forms the same dV
// (bf16(fp32(dv * 1)) = dv) and hence every output of the FP32-dY variant.
//
// HBM-bound streaming: each thread converts 8 consecutive values per step
// (two 16-byte loads, one 16-byte store), grid-stride over the flat array.
#include "common.cuh"
#include "kernels.h"

namespace lora {

__global__ void __launch_bounds__(256) dv_from_f32_kernel(const float4* __restrict__ dy, float alpha, int64_t n8,
                                                          uint4* __restrict__ dv) {
  grid_dependency_wait();   // dY (and the workspace the previous launch used) complete
  grid_dependents_launch();
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const float4 a = __ldcs(dy + 2 * i), b = __ldcs(dy + 2 * i + 1);
    const float v[8] = {__fmul_rn(a.x, alpha), __fmul_rn(a.y, alpha), __fmul_rn(a.z, alpha), __fmul_rn(a.w, alpha),
                        __fmul_rn(b.x, alpha), __fmul_rn(b.y, alpha), __fmul_rn(b.z, alpha), __fmul_rn(b.w, alpha)};
    dv[i] = pack_bf16x8(v);
  }
}

cudaError_t launch_dv_from_f32(const float* dy, float alpha, int64_t n, void* dv, int nsm, cudaStream_t st) {
  const int64_t n8 = n / 8;
  const int64_t want = (n8 + 255) / 256;
  const int grid = int(want < int64_t(nsm) * 8 ? (want > 0 ? want : 1) : int64_t(nsm) * 8);
  return launch_pdl(dv_from_f32_kernel, dim3(grid), dim3(256), 0, st, reinterpret_cast<const float4*>(dy), alpha, n8,
                    static_cast<uint4*>(dv));
}

}  // namespace lora
