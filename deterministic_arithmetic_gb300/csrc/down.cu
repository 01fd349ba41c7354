// down.cu -- the reductions over the long dimension:
//   U  partials: U[m][r]  = sum_k x[m][k] * a[r][k]      (forward "U = X @ A^T")
//   dU partials: dU[m][r] = sum_n dv[m][n] * b[n][r],   dv = bf16(dy * alpha)
// (page "[DSv4][P5-3] shared_grouped_lora_delta: CUDA + Triton, both
// batch-invariant", section "Summary"; dV is formed in shared memory and never
// stored, rounding point "D4").
//
// Work unit = (128-row tile, slice of the reduction dimension). A persistent
// CTA streams the unit's 128 x 64 BF16 input tiles through a TMA/mbarrier
// ring (one pass over the input; each tile lands as two 128 x 32 K-slabs with
// a 64-byte swizzle: measured on GB300, the tensor core reads this layout far
// faster than a 128-byte-swizzled 128 x 64 tile, whose MMA operand fetch
// otherwise adds ~40 cycles per MMA to the streaming time), issues
// four tcgen05 MMAs (M=128, N=RP, K=16) per tile, each into its own fresh TMEM
// accumulator (a "leaf" = one 16-term dot product), and eight epilogue warps
// add the leaves with the canonical pairwise tree in FP32 (round to nearest).
// The unit's result is one FP32 partial per (row, r); a separate combine
// launch finishes the same tree across slices and rounds to BF16.
//
// Warp roles: 0 = TMA producer, 1 = MMA issuer (and TMEM owner),
// 2..9 = epilogue (two warps per TMEM lane quarter, half of the columns each),
// 10..13 = dV transform (dU only).
#include "common.cuh"
#include "kernels.h"

namespace lora {

template <int RP, bool DV>
struct DownCfg {
  static constexpr int kBM = 128, kBK = 64;
  static constexpr int kInBytes = kBM * kBK * 2;     // 16 KB input tile: two [128][32] K-slabs
  static constexpr int kSlabBytes = kInBytes / 2;
  static constexpr int kWBytes = RP * kBK * 2;       // RP x 64 weight tile
  static constexpr int kStageBytes = kInBytes + kWBytes;
  static constexpr int kStages = RP == 64 ? 8 : (RP == 32 ? 9 : 10);
  static constexpr int kLeaves = kBK / 16;
  static constexpr int kGroupCols = kLeaves * RP;
  static constexpr int kGroups = 512 / kGroupCols;
  static constexpr int kSlice = down_slice(RP);
  static constexpr int kGS = kSlice / kBK;            // leaf groups per slice (power of two)
  static constexpr int kLevels = kGS == 16 ? 4 : (kGS == 8 ? 3 : (kGS == 4 ? 2 : (kGS == 2 ? 1 : 0)));
  static constexpr int kEpiWarps = 8, kXfWarps = DV ? 4 : 0;
  static constexpr int kThreads = 32 * (2 + kEpiWarps + kXfWarps);
  static constexpr int kCPT = RP / 2;                 // columns per epilogue thread
  static constexpr int kCH = kCPT < 16 ? kCPT : 16;   // columns per TMEM load batch
  static constexpr int kWSpan = DV ? RP * 2 : 128;    // swizzle span of the weight tile
  static constexpr int kPrefetch = 8;                 // input tiles warmed in L2 before the dependency wait
  static constexpr int kNumBars = 3 * kStages + 2 * kGroups + 2;
  static constexpr size_t kSmem = size_t(kStages) * kStageBytes + 1024 + kNumBars * 8 + 16;
  static_assert((1 << kLevels) == kGS, "slice must hold a power-of-two number of tiles");
  static_assert(kGroups >= 2, "TMEM ring too shallow");
  static_assert(kSmem < 256 * 1024, "descriptor start addresses must fit their 14-bit field");
};

// GR: a grouped launch (several sites); otherwise the table holds one site, read at fixed offsets
template <int RP, bool DV, bool GR>
__global__ void __launch_bounds__(DownCfg<RP, DV>::kThreads, 1)
    down_kernel(const __grid_constant__ Sites<DownSite, GR ? kMaxSites : 1> args, uint32_t* status) {
  using C = DownCfg<RP, DV>;
  // site of unit u (sites are few and ordered by first unit)
  auto site = [&](int u) -> const DownSite& {
    if constexpr (!GR) return args.s[0];
    int i = 0;
    while (i + 1 < args.n && u >= args.s[i + 1].u0) ++i;
    return args.s[i];
  };
  const int total = args.total;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;                      // 1024-byte aligned tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + (base - raw) + size_t(C::kStages) * C::kStageBytes);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto ready = [&](int s) { return bar0 + 8u * (C::kStages + s); };
  auto empty = [&](int s) { return bar0 + 8u * (2 * C::kStages + s); };
  auto tfull = [&](int g) { return bar0 + 8u * (3 * C::kStages + g); };
  auto tempty = [&](int g) { return bar0 + 8u * (3 * C::kStages + C::kGroups + g); };
  const uint32_t drain = bar0 + 8u * (3 * C::kStages + 2 * C::kGroups);
  const uint32_t never = drain + 8u;   // completed by nothing (the stall test hook waits on it)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(ready(s), C::kXfWarps > 0 ? C::kXfWarps : 1);
      mbar_init(empty(s), 1);
    }
    for (int g = 0; g < C::kGroups; ++g) {
      mbar_init(tfull(g), 1);
      mbar_init(tempty(g), C::kEpiWarps);
    }
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0u;
    mbar_fence_init();
    for (int i = 0; i < (GR ? args.n : 1); ++i) {
      prefetch_map(&args.s[i].in);
      prefetch_map(&args.s[i].w);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0 && int(blockIdx.x) < total) {
    // the first input tiles of this CTA's first unit, into L2 while the predecessor drains
    const DownSite& S = site(blockIdx.x);
    const int lu = int(blockIdx.x) - S.u0;
    const int mt = lu % S.n_mt, k0 = (lu / S.n_mt) * C::kSlice;
    const int nkb = min((min(S.Kred - k0, C::kSlice) + C::kBK - 1) / C::kBK, C::kPrefetch);
    for (int kb = 0; kb < nkb; ++kb) {
      tma_prefetch_l2(&S.in, k0 + kb * C::kBK, mt * C::kBM);
      tma_prefetch_l2(&S.in, k0 + kb * C::kBK + 32, mt * C::kBM);
    }
  }
  grid_dependency_wait();      // predecessor done: its outputs are this kernel's inputs
  grid_dependents_launch();
  const Abort ab = make_abort(abort_flag, status);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      if (stall_requested(status, kKindDown)) stall_wait(never, ab, 9);   // test hook: a wait that runs out
      const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_last();
      Ring r;
      uint32_t issued = 0, parities = 0;
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const DownSite& S = site(u);
        const int lu = u - S.u0;
        const int mt = lu % S.n_mt, sl = lu / S.n_mt;
        const int k0 = sl * C::kSlice;
        const int nkb = (min(S.Kred - k0, C::kSlice) + C::kBK - 1) / C::kBK;
        for (int kb = 0; kb < nkb; ++kb) {
          if (wait(empty(r.idx), r.phase ^ 1u, ab, 1)) {
            const uint32_t st = base + r.idx * C::kStageBytes;
            const int k = k0 + kb * C::kBK;
            mbar_expect_tx(full(r.idx), C::kStageBytes);
            tma_load(st, &S.in, full(r.idx), k, mt * C::kBM, pol_stream);                     // k .. k+31
            tma_load(st + C::kSlabBytes, &S.in, full(r.idx), k + 32, mt * C::kBM, pol_stream);  // k+32 .. k+63
            if (DV) tma_load(st + C::kInBytes, &S.w, full(r.idx), 0, k, pol_keep);   // b[n][r], n = k..k+63
            else tma_load(st + C::kInBytes, &S.w, full(r.idx), k, 0, pol_keep);      // a[r][k..k+63]
            issued |= 1u << r.idx;
            parities = (parities & ~(1u << r.idx)) | (r.phase << r.idx);
          }
          r.next<C::kStages>();
        }
      }
      // never leave with a copy in flight into this CTA's shared memory
      for (int s = 0; s < C::kStages; ++s)
        if (issued & (1u << s)) wait_drain(full(s), (parities >> s) & 1u, ab, 2);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    // The whole warp follows the schedule, one elected lane issues; operand
    // descriptors are built once for stage 0 and advanced by the stage offset.
    constexpr uint32_t idesc = idesc_bf16(128, RP, 0, DV ? 1 : 0);
    constexpr uint32_t w_layout = layout_for_span(C::kWSpan);
    uint64_t adesc[C::kLeaves], wdesc[C::kLeaves];
#pragma unroll
    for (int j = 0; j < C::kLeaves; ++j) {
      // input slab j/2: K-major, rows of 64 bytes, 64-byte swizzle, 8-row groups 512 bytes
      // apart; K step j = +32 bytes inside the slab's swizzle atom
      adesc[j] = smem_desc(base + (j >> 1) * C::kSlabBytes + 32u * (j & 1), 16u, 512u, kLayoutSW64);
      if (DV)   // b tile [64 n][RP]: MN-major (r contiguous), 8-row groups of one swizzle span
        wdesc[j] = smem_desc(base + C::kInBytes + j * 16u * C::kWSpan, 8u * C::kWSpan, 8u * C::kWSpan, w_layout);
      else      // a tile [RP][64 k]: K-major, 128-byte swizzle
        wdesc[j] = smem_desc(base + C::kInBytes + 32u * j, 16u, 1024u, kLayoutSW128);
    }
    Ring r, g;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const DownSite& S = site(u);
      const int sl = (u - S.u0) / S.n_mt;
      const int k0 = sl * C::kSlice;
      const int nkb = (min(S.Kred - k0, C::kSlice) + C::kBK - 1) / C::kBK;
      for (int kb = 0; kb < nkb; ++kb) {
        bool ok = wait(DV ? ready(r.idx) : full(r.idx), r.phase, ab, 3);
        ok = __all_sync(0xffffffffu, ok && wait(tempty(g.idx), g.phase ^ 1u, ab, 4));
        if (ok) {
          tc_fence_after();
          const uint32_t off = r.idx * C::kStageBytes;
          const uint32_t d = tmem + g.idx * C::kGroupCols;
#pragma unroll
          for (int j = 0; j < C::kLeaves; ++j)   // fresh accumulator: one leaf
            if (elect_one()) mma_bf16(d + j * RP, desc_advance(adesc[j], off), desc_advance(wdesc[j], off), idesc, 0u);
          if (elect_one()) {
            mma_commit(empty(r.idx));
            mma_commit(tfull(g.idx));
          }
          __syncwarp();
        }
        r.next<C::kStages>();
        g.next<C::kGroups>();
      }
    }
    if (elect_one()) mma_commit(drain);   // all MMAs issued above have completed ...
    __syncwarp();
    wait_drain(drain, 0u, ab, 5);          // ... before TMEM is released
  } else if (warp < 2 + C::kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                            // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;                     // column half
    const uint32_t tbase = tmem + (uint32_t(q * 32) << 16) + h * C::kCPT;
    Ring g;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const DownSite& S = site(u);
      const int lu = u - S.u0;
      const int mt = lu % S.n_mt, sl = lu / S.n_mt;
      const int k0 = sl * C::kSlice;
      const int nkb = (min(S.Kred - k0, C::kSlice) + C::kBK - 1) / C::kBK;
      float stack[C::kLevels > 0 ? C::kLevels : 1][C::kCPT];
      float node[C::kCPT];
      bool ok_all = true;
#pragma unroll
      for (int i = 0; i < C::kGS; ++i) {
        if (i < nkb) {
          const bool ok = __all_sync(0xffffffffu, wait(tfull(g.idx), g.phase, ab, 6));   // warp-uniform: tcgen05.ld is .aligned
          ok_all = ok_all && ok;
          tc_fence_after();
#pragma unroll
          for (int ch = 0; ch < C::kCPT / C::kCH; ++ch) {
            uint32_t v[C::kLeaves][C::kCH / 8][8];
            if (ok) {
#pragma unroll
              for (int j = 0; j < C::kLeaves; ++j)
#pragma unroll
                for (int b8 = 0; b8 < C::kCH / 8; ++b8)
                  tmem_ld8(tbase + g.idx * C::kGroupCols + j * RP + ch * C::kCH + b8 * 8, v[j][b8]);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int j = 0; j < C::kLeaves; ++j)
#pragma unroll
                for (int b8 = 0; b8 < C::kCH / 8; ++b8)
#pragma unroll
                  for (int e = 0; e < 8; ++e) v[j][b8][e] = 0u;
            }
#pragma unroll
            for (int j = 0; j < C::kLeaves; ++j)
#pragma unroll
              for (int b8 = 0; b8 < C::kCH / 8; ++b8) reg_fence(v[j][b8]);
#pragma unroll
            for (int c = 0; c < C::kCH; ++c)
              node[ch * C::kCH + c] = tree4(__uint_as_float(v[0][c / 8][c % 8]), __uint_as_float(v[1][c / 8][c % 8]),
                                            __uint_as_float(v[2][c / 8][c % 8]), __uint_as_float(v[3][c / 8][c % 8]));
          }
          tc_fence_before();
          __syncwarp();
          if (ok && lane == 0) mbar_arrive(tempty(g.idx));
          g.next<C::kGroups>();
        } else {
#pragma unroll
          for (int c = 0; c < C::kCPT; ++c) node[c] = 0.0f;   // zero leaves: neutral in the tree
        }
        // canonical pairwise tree over the slice's groups: merge once per trailing one of i
#pragma unroll
        for (int l = 0; l < C::kLevels; ++l) {
          if (((i >> l) & 1) == 0) {
#pragma unroll
            for (int c = 0; c < C::kCPT; ++c) stack[l][c] = node[c];
            break;
          }
#pragma unroll
          for (int c = 0; c < C::kCPT; ++c) node[c] = __fadd_rn(stack[l][c], node[c]);
        }
      }
      // after the last group (i = kGS - 1, all ones) `node` holds the slice sum
      const int row = mt * C::kBM + q * 32 + lane;
      if (ok_all && row < S.M) {
        float* __restrict__ part = S.part;
        float4* dst = reinterpret_cast<float4*>(part + (size_t(sl) * S.M + row) * RP + h * C::kCPT);
#pragma unroll
        for (int c = 0; c < C::kCPT; c += 4) dst[c / 4] = make_float4(node[c], node[c + 1], node[c + 2], node[c + 3]);
      }
    }
  } else {
    // ---------------------------------------------------- dV = bf16(dY*alpha)
    const int t = threadIdx.x - 32 * (2 + C::kEpiWarps);   // 0..127
    Ring r;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const DownSite& S = site(u);
      const float alpha = S.alpha;
      const uint32_t a2 = pow2_bf16x2(alpha);
      const int sl = (u - S.u0) / S.n_mt;
      const int k0 = sl * C::kSlice;
      const int nkb = (min(S.Kred - k0, C::kSlice) + C::kBK - 1) / C::kBK;
      for (int kb = 0; kb < nkb; ++kb) {
        if (wait(full(r.idx), r.phase, ab, 7)) {
          uint4* tile = reinterpret_cast<uint4*>(smem_raw + (base - raw) + size_t(r.idx) * C::kStageBytes);
#pragma unroll
          for (int e = 0; e < C::kInBytes / 16 / 128; ++e) tile[t + 128 * e] = dv_bf16x8(tile[t + 128 * e], alpha, a2);
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) mbar_arrive(ready(r.idx));
        }
        r.next<C::kStages>();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int RP, bool DV, bool GR>
static cudaError_t launch_one(DownArgs& args, uint32_t* status, int grid, cudaStream_t st) {
  using C = DownCfg<RP, DV>;
  int u0 = 0;
  for (int i = 0; i < args.n; ++i) {
    DownSite& s = args.s[i];
    s.n_mt = int(ceil_div(s.M, C::kBM));
    s.n_sl = int(ceil_div(s.Kred, C::kSlice));
    s.u0 = u0;
    u0 += s.n_mt * s.n_sl;
  }
  args.total = u0;
  if constexpr (GR) return launch_pdl(down_kernel<RP, DV, GR>, dim3(grid), dim3(C::kThreads), C::kSmem, st, args, status);
  else return launch_pdl(down_kernel<RP, DV, GR>, dim3(grid), dim3(C::kThreads), C::kSmem, st, first_site(args), status);
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
  cudaError_t e = cudaFuncSetAttribute(down_kernel<RP, DV, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(DownCfg<RP, DV>::kSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(down_kernel<RP, DV, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(DownCfg<RP, DV>::kSmem));
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
