// wgrad.cu -- the weight gradients, reductions over the batch rows m:
//   dA partials: dA[r][k] = sum_m du[m][r] * x[m][k]           ("dA = dU^T @ X")
//   dB partials: dB[n][r] = sum_m dv[m][n] * u[m][r],  dv = bf16(dy * alpha)   ("dB = dV^T @ U")
// (page "[DSv4][P5-3] shared_grouped_lora_delta: CUDA + Triton, both
// batch-invariant", section "Summary".) These are the worst-shaped GEMMs of
// the LoRA step (page "Independent from-scratch Qwen-14B step
// reimplementation ...", section "Finding 2"): a rank-R output reduced over
// every row of the batch. Here the batch is cut into fixed 256-row chunks
// (never a function of M), each chunk leaves one FP32 partial, and a combine
// launch adds the chunk partials with the canonical pairwise tree.
//
// Work unit = (128-column tile of X or dY, 256-row chunk). Each stage brings
// 64 rows: two 64x64 BF16 boxes of the wide operand (read once, 128-byte
// swizzle) and the 64 x RP slice of du / u. The tensor core computes
// D[col][r] += sum over 16 rows, with both operands MN-major in shared memory
// (M=128 columns, N=RP, K=16 rows); every MMA is a fresh leaf.
//
// Warp roles: 0 = TMA producer, 1 = MMA issuer (TMEM owner), 2..9 = epilogue,
// 10..13 = dV transform (dB only).
#include "common.cuh"
#include "kernels.h"

namespace lora {

template <int RP, bool DV>
struct WgCfg {
  static constexpr int kBC = 128, kBR = 64;
  static constexpr int kInBytes = 2 * 64 * 64 * 2;   // two [64 rows][64 cols] boxes
  static constexpr int kGBytes = kBR * RP * 2;
  static constexpr int kStageBytes = kInBytes + kGBytes;
  static constexpr int kStages = RP == 64 ? 8 : (RP == 32 ? 9 : 10);
  static constexpr int kLeaves = kBR / 16;
  static constexpr int kGroupCols = kLeaves * RP;
  static constexpr int kGroups = 512 / kGroupCols;
  static constexpr int kGS = kWgradChunk / kBR;       // 4 stages per chunk
  static constexpr int kLevels = 2;
  static constexpr int kEpiWarps = 8, kXfWarps = DV ? 4 : 0;
  static constexpr int kThreads = 32 * (2 + kEpiWarps + kXfWarps);
  static constexpr int kCPT = RP / 2;
  static constexpr int kCH = kCPT < 16 ? kCPT : 16;
  static constexpr int kGSpan = RP * 2;
  static constexpr int kNumBars = 3 * kStages + 2 * kGroups + 2;
  static constexpr size_t kSmem = size_t(kStages) * kStageBytes + 1024 + kNumBars * 8 + 16;
  static_assert((1 << kLevels) == kGS, "chunk must hold a power-of-two number of stages");
  static_assert(kSmem < 256 * 1024, "descriptor start addresses must fit their 14-bit field");
};

// GR: a grouped launch (several sites); otherwise the table holds one site, read at fixed offsets
template <int RP, bool DV, bool GR>
__global__ void __launch_bounds__(WgCfg<RP, DV>::kThreads, 1)
    wgrad_kernel(const __grid_constant__ Sites<WgSite, GR ? kMaxSites : 1> args, uint32_t* status) {
  using C = WgCfg<RP, DV>;
  // site of unit u (sites are few and ordered by first unit)
  auto site = [&](int u) -> const WgSite& {
    if constexpr (!GR) return args.s[0];
    int i = 0;
    while (i + 1 < args.n && u >= args.s[i + 1].u0) ++i;
    return args.s[i];
  };
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
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
      prefetch_map(&args.s[i].g);
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
  const int total = args.total;
  auto stages_of = [&](const WgSite& P, int ch) {
    return (min(P.M - ch * kWgradChunk, kWgradChunk) + C::kBR - 1) / C::kBR;
  };
  // The wide operand (X or dY) is an input of the call, which no earlier kernel of the call
  // writes: the first ring stages' copies of it are issued before waiting for the predecessor,
  // so the stream starts while the predecessor's last CTAs finish. (The du / u rows, which the
  // predecessor may have written, are copied only after the wait.)
  int pre = 0;                 // stages whose wide-operand copies are in flight
  if (warp == 0 && lane == 0) {
    const uint64_t pol_stream = policy_evict_first();
    for (int u = blockIdx.x; u < total && pre < C::kStages; u += gridDim.x) {
      const WgSite& P = site(u);
      const int ct = (u - P.u0) % P.n_ct, ch = (u - P.u0) / P.n_ct;
      for (int kb = 0; kb < stages_of(P, ch) && pre < C::kStages; ++kb, ++pre) {
        const uint32_t st = base + pre * C::kStageBytes;
        const int m = ch * kWgradChunk + kb * C::kBR;
        mbar_expect_tx(full(pre), C::kStageBytes);
        tma_load(st, &P.in, full(pre), ct * C::kBC, m, pol_stream);
        tma_load(st + C::kInBytes / 2, &P.in, full(pre), ct * C::kBC + 64, m, pol_stream);
      }
    }
  }
  grid_dependency_wait();      // predecessor done: its outputs are this kernel's inputs
  grid_dependents_launch();
  const Abort ab = make_abort(abort_flag, status);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      if (stall_requested(status, kKindWgrad)) stall_wait(never, ab, 29);   // test hook: a wait that runs out
      const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_last();
      Ring r;
      uint32_t issued = 0, parities = 0;
      int k = 0;               // stage count of this CTA
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const WgSite& P = site(u);
        const int ct = (u - P.u0) % P.n_ct, ch = (u - P.u0) / P.n_ct;
        const int ns = stages_of(P, ch);
        for (int kb = 0; kb < ns; ++kb, ++k) {
          if (k < pre) {         // first pass over the ring: wide operand already in flight
            const uint32_t st = base + r.idx * C::kStageBytes;
            tma_load(st + C::kInBytes, &P.g, full(r.idx), 0, ch * kWgradChunk + kb * C::kBR, pol_keep);
            issued |= 1u << r.idx;
            parities = (parities & ~(1u << r.idx)) | (r.phase << r.idx);
          } else if (wait(empty(r.idx), r.phase ^ 1u, ab, 21)) {
            const uint32_t st = base + r.idx * C::kStageBytes;
            const int m = ch * kWgradChunk + kb * C::kBR;
            mbar_expect_tx(full(r.idx), C::kStageBytes);
            tma_load(st, &P.in, full(r.idx), ct * C::kBC, m, pol_stream);
            tma_load(st + C::kInBytes / 2, &P.in, full(r.idx), ct * C::kBC + 64, m, pol_stream);
            tma_load(st + C::kInBytes, &P.g, full(r.idx), 0, m, pol_keep);
            issued |= 1u << r.idx;
            parities = (parities & ~(1u << r.idx)) | (r.phase << r.idx);
          }
          r.next<C::kStages>();
        }
      }
      for (int s = 0; s < C::kStages; ++s)
        if (issued & (1u << s)) wait_drain(full(s), (parities >> s) & 1u, ab, 22);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    // The whole warp follows the schedule, one elected lane issues; operand
    // descriptors are built once for stage 0 and advanced by the stage offset.
    constexpr uint32_t idesc = idesc_bf16(128, RP, 1, 1);
    constexpr uint32_t g_layout = layout_for_span(C::kGSpan);
    uint64_t adesc[C::kLeaves], gdesc[C::kLeaves];
#pragma unroll
    for (int j = 0; j < C::kLeaves; ++j) {
      // wide operand, transposed view: MN-major (columns contiguous), 128-byte swizzle,
      // 64-column blocks 8 KB apart, 8-row groups 1 KB apart; K step = 16 rows
      adesc[j] = smem_desc(base + j * 2048u, 8192u, 1024u, kLayoutSW128);
      // du / u rows [64][RP]: MN-major (r contiguous), one swizzle span per row
      gdesc[j] = smem_desc(base + C::kInBytes + j * 16u * C::kGSpan, 8u * C::kGSpan, 8u * C::kGSpan, g_layout);
    }
    Ring r, g;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const WgSite& P = site(u);
      const int ch = (u - P.u0) / P.n_ct;
      const int ns = stages_of(P, ch);
      for (int kb = 0; kb < ns; ++kb) {
        bool ok = wait(DV ? ready(r.idx) : full(r.idx), r.phase, ab, 23);
        ok = __all_sync(0xffffffffu, ok && wait(tempty(g.idx), g.phase ^ 1u, ab, 24));
        if (ok) {
          tc_fence_after();
          const uint32_t off = r.idx * C::kStageBytes;
          const uint32_t d = tmem + g.idx * C::kGroupCols;
          if (elect_one()) {   // one lane issues the stage's MMAs back to back
#pragma unroll
            for (int j = 0; j < C::kLeaves; ++j)
              mma_bf16(d + j * RP, desc_advance(adesc[j], off), desc_advance(gdesc[j], off), idesc, 0u);
            mma_commit(empty(r.idx));
            mma_commit(tfull(g.idx));
          }
          __syncwarp();
        }
        r.next<C::kStages>();
        g.next<C::kGroups>();
      }
    }
    if (elect_one()) mma_commit(drain);
    __syncwarp();
    wait_drain(drain, 0u, ab, 25);
  } else if (warp < 2 + C::kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const uint32_t tbase = tmem + (uint32_t(q * 32) << 16) + h * C::kCPT;
    Ring g;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const WgSite& P = site(u);
      const int ct = (u - P.u0) % P.n_ct, ch = (u - P.u0) / P.n_ct;
      const int ns = stages_of(P, ch);
      const int Cw = P.Cw;
      float stack[C::kLevels][C::kCPT];
      float node[C::kCPT];
      bool ok_all = true;
#pragma unroll
      for (int i = 0; i < C::kGS; ++i) {
        if (i < ns) {
          const bool ok = __all_sync(0xffffffffu, wait(tfull(g.idx), g.phase, ab, 26));
          ok_all = ok_all && ok;
          tc_fence_after();
#pragma unroll
          for (int chk = 0; chk < C::kCPT / C::kCH; ++chk) {
            uint32_t v[C::kLeaves][C::kCH / 8][8];
#pragma unroll
            for (int j = 0; j < C::kLeaves; ++j)
#pragma unroll
              for (int b8 = 0; b8 < C::kCH / 8; ++b8)
#pragma unroll
                for (int e = 0; e < 8; ++e) v[j][b8][e] = 0u;
            if (ok) {
#pragma unroll
              for (int j = 0; j < C::kLeaves; ++j)
#pragma unroll
                for (int b8 = 0; b8 < C::kCH / 8; ++b8)
                  tmem_ld8(tbase + g.idx * C::kGroupCols + j * RP + chk * C::kCH + b8 * 8, v[j][b8]);
              tmem_ld_wait();
            }
#pragma unroll
            for (int j = 0; j < C::kLeaves; ++j)
#pragma unroll
              for (int b8 = 0; b8 < C::kCH / 8; ++b8) reg_fence(v[j][b8]);
#pragma unroll
            for (int c = 0; c < C::kCH; ++c)
              node[chk * C::kCH + c] =
                  tree4(__uint_as_float(v[0][c / 8][c % 8]), __uint_as_float(v[1][c / 8][c % 8]),
                        __uint_as_float(v[2][c / 8][c % 8]), __uint_as_float(v[3][c / 8][c % 8]));
          }
          tc_fence_before();
          __syncwarp();
          if (ok && lane == 0) mbar_arrive(tempty(g.idx));
          g.next<C::kGroups>();
        } else {
#pragma unroll
          for (int c = 0; c < C::kCPT; ++c) node[c] = 0.0f;
        }
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
      const int col = ct * C::kBC + q * 32 + lane;
      if (ok_all && col < Cw) {
        float* __restrict__ part = P.part;
        float* dst = part + size_t(ch) * RP * Cw + size_t(h * C::kCPT) * Cw + col;
#pragma unroll
        for (int c = 0; c < C::kCPT; ++c) dst[size_t(c) * Cw] = node[c];
      }
    }
  } else {
    // ---------------------------------------------------- dV = bf16(dY*alpha)
    const int t = threadIdx.x - 32 * (2 + C::kEpiWarps);
    Ring r;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const WgSite& P = site(u);
      const float alpha = P.alpha;
      const uint32_t a2 = pow2_bf16x2(alpha);
      const int ch = (u - P.u0) / P.n_ct;
      const int ns = stages_of(P, ch);
      for (int kb = 0; kb < ns; ++kb) {
        if (wait(full(r.idx), r.phase, ab, 27)) {
          if (!dv_is_dy(alpha)) {
            uint4* tile = reinterpret_cast<uint4*>(smem_raw + (base - raw) + size_t(r.idx) * C::kStageBytes);
#pragma unroll
            for (int e = 0; e < C::kInBytes / 16 / 128; ++e) tile[t + 128 * e] = dv_bf16x8(tile[t + 128 * e], alpha, a2);
            fence_proxy_async();
          }
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

template <int RP, bool DV>
static cudaError_t launch_one(WgArgs& args, uint32_t* status, int grid, cudaStream_t st) {
  using C = WgCfg<RP, DV>;
  int u0 = 0;
  for (int i = 0; i < args.n; ++i) {
    WgSite& s = args.s[i];
    s.n_ct = int(ceil_div(s.Cw, C::kBC));
    s.n_ch = int(ceil_div(s.M, kWgradChunk));
    s.u0 = u0;
    u0 += s.n_ct * s.n_ch;
  }
  args.total = u0;
  if (args.n > 1)
    return launch_pdl(wgrad_kernel<RP, DV, true>, dim3(grid), dim3(C::kThreads), C::kSmem, st, args, status);
  return launch_pdl(wgrad_kernel<RP, DV, false>, dim3(grid), dim3(C::kThreads), C::kSmem, st, first_site(args), status);
}

cudaError_t launch_wgrad(int RP, bool dv, WgArgs& args, uint32_t* status, int grid, cudaStream_t st) {
  if (args.n < 1 || args.n > kMaxSites) return cudaErrorInvalidValue;
  switch (RP * 2 + (dv ? 1 : 0)) {
    case 32: return launch_one<16, false>(args, status, grid, st);
    case 33: return launch_one<16, true>(args, status, grid, st);
    case 64: return launch_one<32, false>(args, status, grid, st);
    case 65: return launch_one<32, true>(args, status, grid, st);
    case 128: return launch_one<64, false>(args, status, grid, st);
    case 129: return launch_one<64, true>(args, status, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int RP, bool DV>
static cudaError_t prep_one() {
  cudaError_t e = cudaFuncSetAttribute(wgrad_kernel<RP, DV, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(WgCfg<RP, DV>::kSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(wgrad_kernel<RP, DV, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(WgCfg<RP, DV>::kSmem));
}

cudaError_t prepare_wgrad() {
  cudaError_t e;
  if ((e = prep_one<16, false>()) != cudaSuccess) return e;
  if ((e = prep_one<16, true>()) != cudaSuccess) return e;
  if ((e = prep_one<32, false>()) != cudaSuccess) return e;
  if ((e = prep_one<32, true>()) != cudaSuccess) return e;
  if ((e = prep_one<64, false>()) != cudaSuccess) return e;
  return prep_one<64, true>();
}

}  // namespace lora
