// up.cu -- the up-projection kernel (dY_lora and dX): one launch of the phase
// in up_phase.cuh, units dealt out round robin. Warp roles and numerics:
// up_phase.cuh.
#include "up_phase.cuh"

namespace lora {

template <int RP, bool DX, bool YBF, bool GR>
__global__ void __launch_bounds__(UpCfg<RP, DX>::kWarps * 32, 1)
    up_kernel(const __grid_constant__ Sites<UpSite, GR ? kMaxSites : 1> args, uint32_t* status) {
  using P = UpPhase<RP, DX, YBF, GR>;
  using C = typename P::C;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + C::kArea);
  const typename P::Bars B{smem_u32(bars)};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  if (threadIdx.x == 0) {
    P::init(B, args);
    *abort_flag = 0u;
    mbar_fence_init();
  }
  if (warp_id() == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dependency_wait();      // predecessor done: its outputs are this kernel's inputs
  grid_dependents_launch();
  const Abort ab = make_abort(abort_flag, status);
  P::run(args, gbase, base, B, tmem, ab, status, StaticSched{args.total}, RowsDone{});
  tc_fence_before();
  __syncthreads();
  if (warp_id() == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int RP, bool DX>
constexpr size_t up_smem() {
  return UpCfg<RP, DX>::kArea + 1024 + UpCfg<RP, DX>::kNumBars * 8 + 16;
}

template <int RP, bool DX, bool YBF, bool GR>
static cudaError_t launch_one(UpArgs& args, uint32_t* status, int grid, cudaStream_t st) {
  using C = UpCfg<RP, DX>;
  up_units_of<RP>(args);
  if constexpr (GR)
    return launch_pdl(up_kernel<RP, DX, YBF, GR>, dim3(grid), dim3(C::kWarps * 32), up_smem<RP, DX>(), st, args,
                      status);
  else
    return launch_pdl(up_kernel<RP, DX, YBF, GR>, dim3(grid), dim3(C::kWarps * 32), up_smem<RP, DX>(), st,
                      first_site(args), status);
}

template <int RP, bool DX, bool YBF>
static cudaError_t launch_gr(UpArgs& args, uint32_t* status, int grid, cudaStream_t st) {
  return args.n > 1 ? launch_one<RP, DX, YBF, true>(args, status, grid, st)
                    : launch_one<RP, DX, YBF, false>(args, status, grid, st);
}

cudaError_t launch_up(int RP, bool dx, bool y_bf16, UpArgs& args, uint32_t* status, int grid, cudaStream_t st) {
  if (dx && y_bf16) return cudaErrorInvalidValue;
  if (args.n < 1 || args.n > kMaxSites) return cudaErrorInvalidValue;
  switch (RP * 4 + (dx ? 1 : 0) + (y_bf16 ? 2 : 0)) {
    case 64: return launch_gr<16, false, false>(args, status, grid, st);
    case 65: return launch_gr<16, true, false>(args, status, grid, st);
    case 66: return launch_gr<16, false, true>(args, status, grid, st);
    case 128: return launch_gr<32, false, false>(args, status, grid, st);
    case 129: return launch_gr<32, true, false>(args, status, grid, st);
    case 130: return launch_gr<32, false, true>(args, status, grid, st);
    case 256: return launch_gr<64, false, false>(args, status, grid, st);
    case 257: return launch_gr<64, true, false>(args, status, grid, st);
    case 258: return launch_gr<64, false, true>(args, status, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int RP, bool DX, bool YBF>
static cudaError_t prep_one() {
  static_assert(up_smem<RP, DX>() < 256 * 1024, "descriptor start addresses must fit their 14-bit field");
  cudaError_t e = cudaFuncSetAttribute(up_kernel<RP, DX, YBF, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(up_smem<RP, DX>()));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(up_kernel<RP, DX, YBF, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(up_smem<RP, DX>()));
}

cudaError_t prepare_up() {
  cudaError_t e;
  if ((e = prep_one<16, false, false>()) != cudaSuccess) return e;
  if ((e = prep_one<16, true, false>()) != cudaSuccess) return e;
  if ((e = prep_one<16, false, true>()) != cudaSuccess) return e;
  if ((e = prep_one<32, false, false>()) != cudaSuccess) return e;
  if ((e = prep_one<32, true, false>()) != cudaSuccess) return e;
  if ((e = prep_one<32, false, true>()) != cudaSuccess) return e;
  if ((e = prep_one<64, false, false>()) != cudaSuccess) return e;
  if ((e = prep_one<64, true, false>()) != cudaSuccess) return e;
  return prep_one<64, false, true>();
}

}  // namespace lora
