// dy.cu -- one pass over the upstream gradient for both backward reductions
// that read it (ranks R <= 16):
//   dV = bf16(dY * alpha)                       (formed in shared memory, never stored; "D4")
//   dU partials: dU[m][r] = sum_n dv[m][n] * b[n][r]   over 512-column slices of N
//   dB partials: dB[n][r] = sum_m dv[m][n] * u[m][r]   over 256-row chunks of M
// (page "[DSv4][P5-3] shared_grouped_lora_delta: CUDA + Triton, both
// batch-invariant", section "Summary": "dV = dY * alpha, dU = dV @ B,
// dB = dV^T @ U"; reading dY once is the fusion its "Benchmark" section points
// at: the elementwise dY traffic, not the GEMMs, is where the time goes.)
//
// Work unit = (256-row chunk, 512-column slice). Each stage brings a 128 x 128
// tile of dY as four 128 x 32 K-slabs (64-byte swizzle) plus the 128 rows of b
// and u it meets; four warps turn it into dV in place. The tensor core then
// reads the same bytes two ways: K-major for dU (8 MMAs, M=128 rows, N=16,
// K=16 columns) and MN-major for dB (8 MMAs, M=128 columns, N=16, K=16 rows);
// every MMA is a fresh leaf. Eight epilogue warps add the leaves with the
// canonical pairwise tree: per 128-row tile over the slice's 32 leaves (one
// dU partial), per 128-column tile over the chunk's 16 leaves (one dB partial).
// Slices and chunks hold power-of-two numbers of leaves, so these partials,
// added by the canonical tree over slices (in the dX kernel) and chunks (in the
// combine), give bit for bit the same dU and dB as the separate dU and dB
// kernels used for larger ranks.
//
// Warp roles: 0 = TMA producer, 1 = MMA issuer (TMEM owner), 2..9 = epilogue,
// 10..13 = dV transform.
#include "common.cuh"
#include "kernels.h"

namespace lora {

struct DyCfg {
  static constexpr int RP = 16;
  static constexpr int kBM = 128, kBN = 128;               // dV tile per stage
  static constexpr int kSlabBytes = kBM * 32 * 2;          // [128 rows][32 columns] BF16: 8 KB
  static constexpr int kTileBytes = 4 * kSlabBytes;        // 32 KB
  static constexpr int kWBytes = 128 * RP * 2;             // b rows n0 .. n0+127: 4 KB
  static constexpr int kGBytes = 128 * RP * 2;             // u rows m0 .. m0+127: 4 KB
  static constexpr int kStageBytes = kTileBytes + kWBytes + kGBytes;
  static constexpr int kStages = 5;
  static constexpr int kLeaves = 8;                        // MMAs of K=16 per product per stage
  static constexpr int kGroupCols = 2 * kLeaves * RP;      // dU leaves + dB leaves: 256 TMEM columns
  static constexpr int kGroups = 512 / kGroupCols;
  static constexpr int kSliceTiles = kDySlice / kBN;       // column tiles per unit (1, 2 or 4)
  static constexpr int kSliceLevels = kSliceTiles == 4 ? 2 : (kSliceTiles == 2 ? 1 : 0);
  static constexpr int kChunkTiles = kDyChunk / kBM;       // 2 row tiles per unit
  static constexpr int kPrefetch = 4;                      // dY tiles warmed in L2 before the dependency wait
  static constexpr int kEpiWarps = 8, kXfWarps = 4;
  static constexpr int kThreads = 32 * (2 + kEpiWarps + kXfWarps);
  static constexpr int kCPT = RP / 2;                      // columns of R per epilogue thread
  static constexpr int kNumBars = 3 * kStages + 2 * kGroups + 2;
  static constexpr size_t kSmem = size_t(kStages) * kStageBytes + 1024 + kNumBars * 8 + 16;
  static_assert((1 << kSliceLevels) == kSliceTiles && kChunkTiles == 2, "epilogue tree shape");
  static_assert(kStageBytes % 1024 == 0, "tiles must stay 1024-byte aligned");
  static_assert(kSmem < 256 * 1024, "descriptor start addresses must fit their 14-bit field");
};

// GR: a grouped launch (several sites); otherwise the table holds one site, read at fixed offsets
template <bool GR>
__global__ void __launch_bounds__(DyCfg::kThreads, 1)
    dy_kernel(const __grid_constant__ Sites<DySite, GR ? kMaxSites : 1> args, uint32_t* status) {
  // site of unit u (sites are few and ordered by first unit)
  auto site = [&](int u) -> const DySite& {
    if constexpr (!GR) return args.s[0];
    int i = 0;
    while (i + 1 < args.n && u >= args.s[i + 1].u0) ++i;
    return args.s[i];
  };
  using C = DyCfg;
  constexpr int RP = C::RP;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + size_t(C::kStages) * C::kStageBytes);
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
      mbar_init(ready(s), C::kXfWarps);
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
      prefetch_map(&args.s[i].dy);
      prefetch_map(&args.s[i].b);
      prefetch_map(&args.s[i].u);
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
  // valid column tiles of a slice and row tiles of a chunk (ragged N and M)
  auto n_tiles = [&](const DySite& P, int sl) { return (min(P.N - sl * kDySlice, kDySlice) + C::kBN - 1) / C::kBN; };
  auto r_tiles = [&](const DySite& P, int ch) { return (min(P.M - ch * kDyChunk, kDyChunk) + C::kBM - 1) / C::kBM; };
  if (threadIdx.x == 0 && int(blockIdx.x) < total) {
    // the first dY tiles of this CTA's first unit, into L2 while the predecessor drains
    const DySite& P = site(blockIdx.x);
    const int sl = (int(blockIdx.x) - P.u0) % P.n_sl, ch = (int(blockIdx.x) - P.u0) / P.n_sl;
    const int nnt = n_tiles(P, sl), nrt = r_tiles(P, ch);
    int n = 0;
    for (int i = 0; i < nnt && n < C::kPrefetch; ++i)
      for (int j = 0; j < nrt && n < C::kPrefetch; ++j, ++n)
        for (int q = 0; q < 4; ++q) tma_prefetch_l2(&P.dy, sl * kDySlice + i * C::kBN + 32 * q, ch * kDyChunk + j * C::kBM);
  }
  grid_dependency_wait();      // predecessor done: its outputs are this kernel's inputs
  grid_dependents_launch();
  const Abort ab = make_abort(abort_flag, status);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      if (stall_requested(status, kKindDy)) stall_wait(never, ab, 39);   // test hook: a wait that runs out
      const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_last();
      Ring r;
      uint32_t issued = 0, parities = 0;
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const DySite& P = site(u);
        const int sl = (u - P.u0) % P.n_sl, ch = (u - P.u0) / P.n_sl;
        const int nnt = n_tiles(P, sl), nrt = r_tiles(P, ch);
        for (int i = 0; i < nnt; ++i)
          for (int j = 0; j < nrt; ++j) {
            if (wait(empty(r.idx), r.phase ^ 1u, ab, 31)) {
              const uint32_t st = base + r.idx * C::kStageBytes;
              const int n0 = sl * kDySlice + i * C::kBN, m0 = ch * kDyChunk + j * C::kBM;
              mbar_expect_tx(full(r.idx), C::kStageBytes);
#pragma unroll
              for (int q = 0; q < 4; ++q)                                       // dy[m0..+127][n0+32q..+31]
                tma_load(st + q * C::kSlabBytes, &P.dy, full(r.idx), n0 + 32 * q, m0, pol_stream);
              tma_load(st + C::kTileBytes, &P.b, full(r.idx), 0, n0, pol_keep);               // b[n0..+127][.]
              tma_load(st + C::kTileBytes + C::kWBytes, &P.u, full(r.idx), 0, m0, pol_keep);  // u[m0..+127][.]
              issued |= 1u << r.idx;
              parities = (parities & ~(1u << r.idx)) | (r.phase << r.idx);
            }
            r.next<C::kStages>();
          }
      }
      for (int s = 0; s < C::kStages; ++s)
        if (issued & (1u << s)) wait_drain(full(s), (parities >> s) & 1u, ab, 32);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    // The whole warp follows the schedule; one elected lane issues a stage's MMAs
    // back to back (one election per stage: measured, an election per MMA made
    // the issue ~60 % slower). Operand descriptors are built once for stage 0 and
    // advanced by the stage offset.
    constexpr uint32_t idesc_du = idesc_bf16(128, RP, 0, 1);   // dV K-major, b MN-major
    constexpr uint32_t idesc_db = idesc_bf16(128, RP, 1, 1);   // dV^T MN-major, u MN-major
    uint64_t a_du[C::kLeaves], b_du[C::kLeaves], a_db[C::kLeaves], b_db[C::kLeaves];
#pragma unroll
    for (int j = 0; j < C::kLeaves; ++j) {
      // dU leaf j: columns 16j..16j+15 -> slab j/2, K-major, 64-byte swizzle (8-row groups 512 B apart)
      a_du[j] = smem_desc(base + (j >> 1) * C::kSlabBytes + 32u * (j & 1), 16u, 512u, kLayoutSW64);
      // b rows 16j..16j+15 of [128 n][16 r]: MN-major, 32-byte swizzle (8-row groups 256 B apart)
      b_du[j] = smem_desc(base + C::kTileBytes + j * 512u, 256u, 256u, kLayoutSW32);
      // dB leaf j: rows 16j..16j+15 of the tile seen MN-major: 32-column atoms 8 KB apart (one per
      // slab), rows of 64 bytes, 8-row groups 512 B apart; K step = 16 rows = 1 KB
      a_db[j] = smem_desc(base + j * 1024u, uint32_t(C::kSlabBytes), 512u, kLayoutSW64);
      b_db[j] = smem_desc(base + C::kTileBytes + C::kWBytes + j * 512u, 256u, 256u, kLayoutSW32);
    }
    Ring r, g;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const DySite& P = site(u);
      const int sl = (u - P.u0) % P.n_sl, ch = (u - P.u0) / P.n_sl;
      const int nstages = n_tiles(P, sl) * r_tiles(P, ch);
      for (int k = 0; k < nstages; ++k) {
        bool ok = wait(ready(r.idx), r.phase, ab, 33);
        ok = __all_sync(0xffffffffu, ok && wait(tempty(g.idx), g.phase ^ 1u, ab, 34));
        if (ok) {
          tc_fence_after();
          const uint32_t off = r.idx * C::kStageBytes;
          const uint32_t d = tmem + g.idx * C::kGroupCols;
          if (elect_one()) {   // one lane issues the stage's MMAs back to back
#pragma unroll
            for (int j = 0; j < C::kLeaves; ++j)
              mma_bf16(d + j * RP, desc_advance(a_du[j], off), desc_advance(b_du[j], off), idesc_du, 0u);
#pragma unroll
            for (int j = 0; j < C::kLeaves; ++j)
              mma_bf16(d + C::kLeaves * RP + j * RP, desc_advance(a_db[j], off), desc_advance(b_db[j], off), idesc_db, 0u);
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
    wait_drain(drain, 0u, ab, 35);
  } else if (warp < 2 + C::kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;                        // column half of R
    const uint32_t tq = tmem + (uint32_t(q * 32) << 16) + h * C::kCPT;
    const int tr = q * 32 + lane;                         // TMEM lane: row (dU) or column (dB) within the tile
    Ring g;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const DySite& P = site(u);
      const int sl = (u - P.u0) % P.n_sl, ch = (u - P.u0) / P.n_sl;
      const int nnt = n_tiles(P, sl), nrt = r_tiles(P, ch);
      const int M = P.M, N = P.N;
      float* __restrict__ du_part = P.du_part;
      float* __restrict__ db_part = P.db_part;
      float du_stk[C::kChunkTiles][C::kSliceLevels > 0 ? C::kSliceLevels : 1][C::kCPT];   // per row tile: tree stack
      float db_first[C::kCPT];
      bool ok_all = true;
#pragma unroll
      for (int i = 0; i < C::kSliceTiles; ++i) {
#pragma unroll
        for (int j = 0; j < C::kChunkTiles; ++j) {
          float dun[C::kCPT], dbn[C::kCPT];
          if (i < nnt && j < nrt) {
            const bool ok = __all_sync(0xffffffffu, wait(tfull(g.idx), g.phase, ab, 36));
            ok_all = ok_all && ok;
            tc_fence_after();
            const uint32_t ta = tq + g.idx * C::kGroupCols;
            float x0[8], x1[8];
            leaves4_tree(ta, ok, x0);                             // dU leaves 0..3
            leaves4_tree(ta + 4 * RP, ok, x1);                    // dU leaves 4..7
#pragma unroll
            for (int c = 0; c < C::kCPT; ++c) dun[c] = __fadd_rn(x0[c], x1[c]);
            leaves4_tree(ta + C::kLeaves * RP, ok, x0);           // dB leaves 0..3
            leaves4_tree(ta + C::kLeaves * RP + 4 * RP, ok, x1);  // dB leaves 4..7
#pragma unroll
            for (int c = 0; c < C::kCPT; ++c) dbn[c] = __fadd_rn(x0[c], x1[c]);
            tc_fence_before();
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(tempty(g.idx));
            g.next<C::kGroups>();
          } else {
#pragma unroll
            for (int c = 0; c < C::kCPT; ++c) dun[c] = dbn[c] = 0.0f;   // zero leaves: neutral in the tree
          }
          // dU of row tile j: canonical tree over the slice's column tiles (merge once per trailing
          // one of i); after the last tile `dun` holds the slice's partial
          bool merged = true;
#pragma unroll
          for (int l = 0; l < C::kSliceLevels; ++l) {
            if (((i >> l) & 1) == 0) {
#pragma unroll
              for (int c = 0; c < C::kCPT; ++c) du_stk[j][l][c] = dun[c];
              merged = false;
              break;
            }
#pragma unroll
            for (int c = 0; c < C::kCPT; ++c) dun[c] = __fadd_rn(du_stk[j][l][c], dun[c]);
          }
          if (merged && i == C::kSliceTiles - 1) {
            const int row = ch * kDyChunk + j * C::kBM + tr;
            if (ok_all && j < nrt && row < M) {
              float4* dst = reinterpret_cast<float4*>(du_part + (size_t(sl) * M + row) * RP + h * C::kCPT);
              dst[0] = make_float4(dun[0], dun[1], dun[2], dun[3]);
              dst[1] = make_float4(dun[4], dun[5], dun[6], dun[7]);
            }
          }
          // dB of column tile i: the chunk's two row tiles
          if (j == 0) {
#pragma unroll
            for (int c = 0; c < C::kCPT; ++c) db_first[c] = dbn[c];
          } else {
            const int col = sl * kDySlice + i * C::kBN + tr;
            if (ok_all && i < nnt && col < N) {
              float* dst = db_part + (size_t(ch) * RP + h * C::kCPT) * N + col;
#pragma unroll
              for (int c = 0; c < C::kCPT; ++c) dst[size_t(c) * N] = __fadd_rn(db_first[c], dbn[c]);
            }
          }
        }
      }
    }
  } else {
    // ---------------------------------------------------- dV = bf16(dY*alpha)
    const int t = threadIdx.x - 32 * (2 + C::kEpiWarps);
    Ring r;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const DySite& P = site(u);
      const float alpha = P.alpha;
      const uint32_t a2 = pow2_bf16x2(alpha);
      const int sl = (u - P.u0) % P.n_sl, ch = (u - P.u0) / P.n_sl;
      const int nstages = n_tiles(P, sl) * r_tiles(P, ch);
      for (int k = 0; k < nstages; ++k) {
        if (wait(full(r.idx), r.phase, ab, 37)) {
          if (!dv_is_dy(alpha)) {
            uint4* tile = reinterpret_cast<uint4*>(gbase + size_t(r.idx) * C::kStageBytes);
#pragma unroll
            for (int e = 0; e < C::kTileBytes / 16 / (32 * C::kXfWarps); ++e)
              tile[t + 32 * C::kXfWarps * e] = dv_bf16x8(tile[t + 32 * C::kXfWarps * e], alpha, a2);
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

cudaError_t launch_dy(DyArgs& args, uint32_t* status, int grid, cudaStream_t st) {
  if (args.n < 1 || args.n > kMaxSites) return cudaErrorInvalidValue;
  int u0 = 0;
  for (int i = 0; i < args.n; ++i) {
    DySite& s = args.s[i];
    s.n_sl = int(ceil_div(s.N, kDySlice));
    s.n_ch = int(ceil_div(s.M, kDyChunk));
    s.u0 = u0;
    u0 += s.n_sl * s.n_ch;
  }
  args.total = u0;
  if (args.n > 1) return launch_pdl(dy_kernel<true>, dim3(grid), dim3(DyCfg::kThreads), DyCfg::kSmem, st, args, status);
  return launch_pdl(dy_kernel<false>, dim3(grid), dim3(DyCfg::kThreads), DyCfg::kSmem, st, first_site(args), status);
}

cudaError_t prepare_dy() {
  const cudaError_t e =
      cudaFuncSetAttribute(dy_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(DyCfg::kSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(dy_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(DyCfg::kSmem));
}

}  // namespace lora
