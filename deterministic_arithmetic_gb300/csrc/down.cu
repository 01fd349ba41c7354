// down.cu -- the down-projection kernel (U partials, and dU partials for ranks
// above 16): one launch of the phase in down_phase.cuh, units dealt out round
// robin. Warp roles and numerics: down_phase.cuh.
#include "down_phase.cuh"

namespace lora {

// no-op epilogue hook of a standalone launch
struct NoHook {
  __device__ __forceinline__ void stored(int) {}
};

template <int RP, bool DV, bool GR>
__global__ void __launch_bounds__(DownCfg<RP, DV>::kWarps * 32, 1)
    down_kernel(const __grid_constant__ Sites<DownSite, GR ? kMaxSites : 1> args, uint32_t* status) {
  using P = DownPhase<RP, DV, GR>;
  using C = typename P::C;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;                      // 1024-byte aligned tiles
  uint8_t* gbase = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + C::kStageArea);
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
  if (threadIdx.x == 0) P::warm_l2(args, blockIdx.x);   // into L2 while the predecessor drains
  grid_dependency_wait();      // predecessor done: its outputs are this kernel's inputs
  grid_dependents_launch();
  const Abort ab = make_abort(abort_flag, status);
  const StaticSched sched{args.total};
  NoHook hook;
  P::run(args, gbase, base, B, tmem, ab, status, sched, sched, hook);
  tc_fence_before();
  __syncthreads();
  if (warp_id() == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int RP, bool DV>
constexpr size_t down_smem() {
  return DownCfg<RP, DV>::kStageArea + 1024 + DownCfg<RP, DV>::kNumBars * 8 + 16;
}

template <int RP, bool DV, bool GR>
static cudaError_t launch_one(DownArgs& args, uint32_t* status, int grid, cudaStream_t st) {
  using C = DownCfg<RP, DV>;
  down_units_of<RP>(args);
  if constexpr (GR)
    return launch_pdl(down_kernel<RP, DV, GR>, dim3(grid), dim3(C::kWarps * 32), down_smem<RP, DV>(), st, args, status);
  else
    return launch_pdl(down_kernel<RP, DV, GR>, dim3(grid), dim3(C::kWarps * 32), down_smem<RP, DV>(), st,
                      first_site(args), status);
}

cudaError_t launch_down(int RP, bool dv, DownArgs& args, uint32_t* status, int grid, cudaStream_t st) {
  if (args.n < 1 || args.n > kMaxSites) return cudaErrorInvalidValue;
  const bool gr = args.n > 1;
  switch (RP * 4 + (dv ? 1 : 0) + (gr ? 2 : 0)) {
    case 64: return launch_one<16, false, false>(args, status, grid, st);
    case 65: return launch_one<16, true, false>(args, status, grid, st);
    case 66: return launch_one<16, false, true>(args, status, grid, st);
    case 67: return launch_one<16, true, true>(args, status, grid, st);
    case 128: return launch_one<32, false, false>(args, status, grid, st);
    case 129: return launch_one<32, true, false>(args, status, grid, st);
    case 130: return launch_one<32, false, true>(args, status, grid, st);
    case 131: return launch_one<32, true, true>(args, status, grid, st);
    case 256: return launch_one<64, false, false>(args, status, grid, st);
    case 257: return launch_one<64, true, false>(args, status, grid, st);
    case 258: return launch_one<64, false, true>(args, status, grid, st);
    case 259: return launch_one<64, true, true>(args, status, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int RP, bool DV>
static cudaError_t prep_one() {
  static_assert(down_smem<RP, DV>() < 256 * 1024, "descriptor start addresses must fit their 14-bit field");
  cudaError_t e = cudaFuncSetAttribute(down_kernel<RP, DV, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(down_smem<RP, DV>()));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(down_kernel<RP, DV, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(down_smem<RP, DV>()));
}

cudaError_t prepare_down() {
  cudaError_t e;
  if ((e = prep_one<16, false>()) != cudaSuccess) return e;
  if ((e = prep_one<16, true>()) != cudaSuccess) return e;
  if ((e = prep_one<32, false>()) != cudaSuccess) return e;
  if ((e = prep_one<32, true>()) != cudaSuccess) return e;
  if ((e = prep_one<64, false>()) != cudaSuccess) return e;
  return prep_one<64, true>();
}

}  // namespace lora
