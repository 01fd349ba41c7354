// fwd_fused.cu -- the forward pass of one site in a single launch:
//   U partials (the down phase), U = bf16(tree over the slices) (the rows step),
//   dY_lora = fp32(U @ B^T) * alpha (the up phase)
// (page "[DSv4][P5-3] shared_grouped_lora_delta: CUDA + Triton, both
// batch-invariant", section "Summary"; its review thread asks for GEMM1 and
// GEMM2 in one kernel, with U still stored).
//
// The three steps depend on each other across CTAs: a row tile's U rows need
// all of its slice partials, and a tile of dY_lora needs its U rows. No CTA
// waits at a grid-wide barrier, and no CTA ever waits for work that a CTA not
// yet running holds:
//   - down units are claimed from a ticket counter (QueueSched), so every
//     claimed unit belongs to a running CTA, which finishes it without
//     waiting for anything; a signal warp counts each finished partial into
//     its row tile's `done` word (after a GPU-scope release fence);
//   - a CTA whose down claims have run out claims row tiles from a second
//     counter; every down unit has been claimed by then, so waiting for a
//     tile's `done` count ends; the whole CTA forms the tile's BF16 rows,
//     writes them to u and raises the tile's `ready` flag (release);
//   - then the CTA runs its up units (round robin); every row tile has been
//     claimed by then, so waiting for a `ready` flag ends.
// So a plain launch is enough (no cooperative launch, no assumption about how
// many CTAs are resident). The last CTA to leave puts the control words back
// to zero for the next launch; every CTA leaves once, also when aborting.
// Results are bit for bit those of the down, rows and up kernels: the same
// leaves, the same canonical trees, the same rounding points.
//
// Warp roles: 0..9 the phases' roles (down_phase.cuh, up_phase.cuh), 10 the
// signal warp of the down phase; the rows step uses every thread.
#include "down_phase.cuh"
#include "up_phase.cuh"

namespace lora {

constexpr int kFusedSignalWarp = 10;
constexpr int kFusedWarps = 11;

template <int RP>
struct FusedCfg {
  using D = DownCfg<RP, false>;
  using U = UpCfg<RP, false>;
  static constexpr size_t kArea = D::kStageArea > U::kArea ? D::kStageArea : U::kArea;
  static constexpr int kDownBars = D::kNumBars, kUpBars = U::kNumBars;
  // mbarriers: down phase, up phase, queue (full, free), hand-over ring (done, free)
  static constexpr int kNumBars = kDownBars + kUpBars + 2 * kQueueSlots + 4;
  // after the barriers: queue slots (ints), then tmem slot, abort flag, row-tile broadcast word
  static constexpr size_t kSmem = kArea + 1024 + kNumBars * 8 + kQueueSlots * 4 + 16;
  static_assert(D::kWarps <= kFusedSignalWarp && U::kWarps <= kFusedSignalWarp, "signal warp after the roles");
  static_assert(kSmem < 227 * 1024, "one CTA per SM");
};

// Control words of a fused forward launch (in the workspace's control block; zero between launches).
struct FwdCtl {
  unsigned int* words;   // [0] down tickets, [1] row-tile tickets, [2] CTAs that have left
  uint32_t* done;        // [n_mt] slice partials counted per row tile
  uint32_t* ready;       // [n_mt] rows of the tile written
};

struct FusedFwdArgs {
  Sites<DownSite, 1> down;
  Sites<UpSite, 1> up;
  FwdCtl ctl;
  __nv_bfloat16* u;      // [M][R]
  int R;
};

// Epilogue hook of the down phase: hand the k-th unit's stored partial to the signal warp
// through a two-slot ring (the slot's previous unit must have been taken).
struct HandOver {
  uint32_t done0, free0;   // mbarriers: [2] done (8 epilogue warps), [2] free (signal warp)
  Abort ab;
  __device__ __forceinline__ void stored(int k) {
    wait(free0 + 8u * (k & 1), ((k >> 1) & 1) ^ 1u, ab, 42);
    __syncwarp();
    if (lane_id() == 0) mbar_arrive(done0 + 8u * (k & 1));
  }
};

// Up-phase rows policy: wait for the row tile's ready flag (set by another CTA with a release
// store after its generic writes of u), then order those writes before the TMA loads of u.
struct RowsFlag {
  const uint32_t* flags;   // [n_mt] ready flags
  __device__ __forceinline__ bool ready(const UpSite&, int mt, const Abort& ab) const {
    if (!wait_global_at_least(flags + mt, 1u, ab, 43)) return false;
    fence_proxy_async_global();
    return true;
  }
};

template <int RP, bool YBF>
__global__ void __launch_bounds__(kFusedWarps * 32, 1)
    fwd_fused_kernel(const __grid_constant__ FusedFwdArgs args, uint32_t* status) {
  using F = FusedCfg<RP>;
  using DP = DownPhase<RP, false, false>;
  using UP = UpPhase<RP, false, YBF, false>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + F::kArea);
  const uint32_t bar0 = smem_u32(bars);
  const typename DP::Bars DB{bar0};
  const typename UP::Bars UB{bar0 + 8u * F::kDownBars};
  const uint32_t q0 = bar0 + 8u * (F::kDownBars + F::kUpBars);
  const uint32_t hand0 = q0 + 8u * (2 * kQueueSlots);                  // done[2], free[2]
  volatile int* qid = reinterpret_cast<volatile int*>(bars + F::kNumBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + F::kNumBars) + kQueueSlots;
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile int* bcast = reinterpret_cast<volatile int*>(tmem_slot + 2);
  const QueueRing ring{qid, q0, q0 + 8u * kQueueSlots};
  const DownSite& DS = args.down.s[0];
  const int n_mt = DS.n_mt, S = DS.n_sl;

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    DP::init(DB, args.down);
    UP::init(UB, args.up);
    ring.init(1 + 8 + 1);                            // reader warps: MMA, 8 epilogue, signal
    for (int i = 0; i < 2; ++i) {
      mbar_init(hand0 + 8u * i, 8);                  // done: the 8 epilogue warps
      mbar_init(hand0 + 8u * (2 + i), 1);            // free: the signal warp
    }
    *abort_flag = 0u;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dependency_wait();      // predecessor done (and the previous launch's control words reset)
  grid_dependents_launch();
  const Abort ab = make_abort(abort_flag, status);

  // ------------------------------------------------ down phase (claimed units)
  {
    QueueProducer ps{ring, args.ctl.words + 0, args.down.total, ab, 44};
    QueueReader rs{ring, ab, 45};
    HandOver hook{hand0, hand0 + 16u, ab};
    if (warp == kFusedSignalWarp) {
      // count each stored partial into its row tile's `done` word; every unit is counted, also
      // when the CTA is aborting, so that no other CTA waits for it until its limit
      int k = 0;
      for (int u = rs.first(); u >= 0; u = rs.next(u), ++k) {
        wait(hand0 + 8u * (k & 1), (k >> 1) & 1, ab, 46);
        if (lane == 0) {
          asm volatile("fence.acq_rel.gpu;" ::: "memory");   // the partial before the count
          atomicAdd(args.ctl.done + (u - DS.u0) / S, 1u);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(hand0 + 16u + 8u * (k & 1));
      }
    } else {
      DP::run(args.down, gbase, base, DB, tmem, ab, status, ps, rs, hook);
    }
  }
  tc_fence_before();
  __syncthreads();             // this CTA's down work is finished: shared memory and TMEM are free
  tc_fence_after();

  // ------------------------------------------------ rows step (claimed row tiles)
  const int R = args.R;
  for (;;) {
    if (threadIdx.x == 0) {
      int t = int(atomicAdd(args.ctl.words + 1, 1u));
      if (t < n_mt && !wait_global_at_least(args.ctl.done + t, uint32_t(S), ab, 47)) t = -2 - t;   // aborting
      *bcast = t;
    }
    __syncthreads();
    const int t = *bcast;
    __syncthreads();
    if (t >= n_mt) break;
    const int mt = t >= 0 ? t : -2 - t;
    if (t >= 0) {
      for (int i = threadIdx.x; i < 128 * (R / 8); i += blockDim.x) {
        const int row = mt * 128 + i / (R / 8), g = i % (R / 8);
        if (row < DS.M)
          *reinterpret_cast<uint4*>(args.u + size_t(row) * R + g * 8) =
              slices_to_bf16x8(DS.part + size_t(row) * RP + g * 8, size_t(DS.M) * RP, S);
      }
    }
    __syncthreads();           // every row of the tile written by this CTA ...
    if (threadIdx.x == 0) st_release_gpu(args.ctl.ready + mt, 1u);   // ... before the flag (release)
  }

  // ------------------------------------------------ up phase (round robin)
  UP::run(args.up, gbase, base, UB, tmem, ab, status, StaticSched{args.up.total}, RowsFlag{args.ctl.ready});

  // ------------------------------------------------ leave; the last CTA resets the control words
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    *bcast = atomicAdd(args.ctl.words + 2, 1u) == gridDim.x - 1u ? 1 : 0;
  }
  __syncthreads();
  if (*bcast) {
    for (int i = threadIdx.x; i < n_mt; i += blockDim.x) {
      args.ctl.done[i] = 0u;
      args.ctl.ready[i] = 0u;
    }
    if (threadIdx.x == 0) {
      args.ctl.words[0] = 0u;
      args.ctl.words[1] = 0u;
      args.ctl.words[2] = 0u;
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int RP, bool YBF>
static cudaError_t launch_fused(FusedFwdArgs& a, uint32_t* status, int grid, cudaStream_t st) {
  return launch_pdl(fwd_fused_kernel<RP, YBF>, dim3(grid), dim3(kFusedWarps * 32), FusedCfg<RP>::kSmem, st, a, status);
}

cudaError_t launch_fwd_fused(int RP, bool y_bf16, DownArgs& dargs, UpArgs& uargs, __nv_bfloat16* u, int R,
                             uint32_t* ctl, int nsm, uint32_t* status, cudaStream_t st) {
  if (dargs.n != 1 || uargs.n != 1) return cudaErrorInvalidValue;
  FusedFwdArgs a{};
  switch (RP) {
    case 16: down_units_of<16>(dargs); up_units_of<16>(uargs); break;
    case 32: down_units_of<32>(dargs); up_units_of<32>(uargs); break;
    case 64: down_units_of<64>(dargs); up_units_of<64>(uargs); break;
    default: return cudaErrorInvalidValue;
  }
  if (dargs.s[0].n_mt > kFusedMaxTiles) return cudaErrorInvalidValue;
  a.down = first_site(dargs);
  a.up = first_site(uargs);
  a.ctl.words = ctl;
  a.ctl.done = ctl + 4;
  a.ctl.ready = ctl + 4 + kFusedMaxTiles;
  a.u = u;
  a.R = R;
  const int grid = int(std::max<int64_t>(1, std::min<int64_t>(std::max(a.down.total, a.up.total), nsm)));
  switch (RP * 2 + (y_bf16 ? 1 : 0)) {
    case 32: return launch_fused<16, false>(a, status, grid, st);
    case 33: return launch_fused<16, true>(a, status, grid, st);
    case 64: return launch_fused<32, false>(a, status, grid, st);
    case 65: return launch_fused<32, true>(a, status, grid, st);
    case 128: return launch_fused<64, false>(a, status, grid, st);
    case 129: return launch_fused<64, true>(a, status, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int RP, bool YBF>
static cudaError_t prep_fused_one() {
  return cudaFuncSetAttribute(fwd_fused_kernel<RP, YBF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(FusedCfg<RP>::kSmem));
}

cudaError_t prepare_fwd_fused() {
  cudaError_t e;
  if ((e = prep_fused_one<16, false>()) != cudaSuccess) return e;
  if ((e = prep_fused_one<16, true>()) != cudaSuccess) return e;
  if ((e = prep_fused_one<32, false>()) != cudaSuccess) return e;
  if ((e = prep_fused_one<32, true>()) != cudaSuccess) return e;
  if ((e = prep_fused_one<64, false>()) != cudaSuccess) return e;
  return prep_fused_one<64, true>();
}

}  // namespace lora
