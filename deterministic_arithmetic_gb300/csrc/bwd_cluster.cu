// bwd_cluster.cu -- the backward pass (ranks R <= 16) in one launch of thread-block clusters:
//   dV = bf16(dY * alpha)                          (formed in shared memory, never stored)
//   dU partials: dU[m][r] = sum_n dv[m][n] * b[n][r]   over 512-column slices of N
//   dB partials: dB[n][r] = sum_m dv[m][n] * u[m][r]   per 256-row chunk of M
//   dU rows:     dU = bf16(canonical tree over the slices)
//   dX[m][k]   = fp32(sum_r du[m][r] * a[r][k])
//   dA partials: dA[r][k] = sum_m du[m][r] * x[m][k]   per 256-row chunk of M
// (page "[DSv4][P5-3] shared_grouped_lora_delta: CUDA + Triton, both
// batch-invariant", section "Summary": "dV = dY * alpha, dU = dV @ B,
// dB = dV^T @ U, dX = dU @ A, dA = dU^T @ X"; the combine launch that follows
// adds the chunk partials of dA and dB with the canonical tree over chunks.)
//
// A cluster of CL CTAs owns one 256-row chunk at a time; clusters take chunks
// round robin. CTA rank r of the cluster:
//   phase A: streams the 512-column slices r, r + CL, ... of the chunk's dY
//     rows (128 x 128 tiles), turns each tile into dV in shared memory and
//     reads it twice with the tensor core: K-major for the dU leaves, MN-major
//     for the dB leaves (the fused pass of the standalone dy kernel); stores
//     each slice's dU partial and each 128-column tile's dB chunk partial;
//   the cluster meets (an mbarrier in every peer's shared memory, release /
//     acquire at cluster scope), then every CTA adds all slice partials of the
//     chunk's rows with the canonical tree, rounds to BF16 and keeps the 256
//     dU rows in its shared memory (swizzled, as the tensor core reads them);
//     rank r stores its 256 / CL rows of du;
//   phase C: for its 128-column tiles r, r + CL, ... of K, per 128-row half
//     of the chunk: streams x (128 x 128) and the a columns, and issues the dA
//     leaves (x^T with du, M = 128 columns, K = 16 rows) and the dX expansion
//     (du with a, M = 128 rows, N = 128 columns, K = 16) into one TMEM slot;
//     the epilogue adds the dA leaves (canonical tree over the chunk's 16
//     leaves) into the chunk partial and stores dX with TMA (evict-first).
// The x copies of phase C do not depend on dU, so the producer streams them
// while the cluster meets. Every leaf, tree and rounding point is that of the
// standalone dy, rows, up (dX) and wgrad (dA) kernels: the outputs agree with
// the separate launches bit for bit.
//
// Warp roles: 0 = TMA producer, 1 = MMA issuer (TMEM owner), 2..9 = epilogue,
// 10..13 = dV transform. Stages share one ring of shared-memory slots and one
// ring of two 256-column TMEM slots, in the order the producer fills them.
#include "common.cuh"
#include "kernels.h"

namespace lora {

template <bool PC>
struct BcCfg {
  static constexpr int RP = 16;
  static constexpr int kBM = 128;
  // phase A slot: dY [128][128] as four [128][32] K-slabs (64-byte swizzle), b rows, u rows
  static constexpr int kSlabBytes = kBM * 32 * 2;          // 8 KB
  static constexpr int kTileBytes = 4 * kSlabBytes;        // 32 KB
  static constexpr int kWBytes = 128 * RP * 2;             // 4 KB
  // phase C slot: x [128][128] as two 64-row halves of two [64][64] boxes (128-byte swizzle), a [RP][128]
  static constexpr int kXBytes = 128 * 128 * 2;            // 32 KB
  static constexpr int kABytes = RP * 128 * 2;             // 4 KB
  static constexpr int kSlotBytes = kTileBytes + 2 * kWBytes;   // 40 KB (phase C uses 36 KB)
  static constexpr int kSlots = 4;                         // five measured slower without phase C
  static constexpr int kLeaves = 8;                        // 16-term leaves per 128 of the reduction
  static constexpr int kTCols = 256, kTSlots = 2;          // TMEM ring
  static constexpr int kSliceTiles = kDySlice / 128;       // column tiles per dU slice
  static constexpr int kSliceLevels = kSliceTiles == 4 ? 2 : (kSliceTiles == 2 ? 1 : 0);
  static constexpr int kEpiWarps = 8, kXfWarps = 4;
  static constexpr int kThreads = 32 * (2 + kEpiWarps + kXfWarps);
  static constexpr int kCPT = RP / 2;                      // columns of R per epilogue thread
  static constexpr int kStg = 1, kStgBytes = 32 * 32 * 4;  // dX staging boxes per epilogue warp
  static constexpr int kDuBytes = 2 * kBM * RP * 2;        // the chunk's 256 dU rows: 8 KB
  static constexpr size_t kDuOff = size_t(kSlots) * kSlotBytes;
  static constexpr size_t kStgOff = kDuOff + kDuBytes;
  static constexpr size_t kArea = PC ? kStgOff + size_t(kEpiWarps) * kStg * kStgBytes : kDuOff;
  // mbarriers: slots (full, ready, empty), TMEM (full, empty), dU exchange [2], dU set, drain, never
  static constexpr int kNumBars = 3 * kSlots + 2 * kTSlots + 2 + 1 + 2;
  static constexpr size_t kSmem = kArea + 1024 + kNumBars * 8 + 16;
  static_assert(kSlotBytes % 1024 == 0 && kDuOff % 1024 == 0 && kStgOff % 1024 == 0, "1024-byte aligned tiles");
  static_assert((1 << kSliceLevels) == kSliceTiles && kDyChunk == 2 * kBM && kWgradChunk == kDyChunk, "tree shapes");
  static_assert(kSmem < 227 * 1024, "one CTA per SM");
};

// PC = false: phase A and the dU rows only (each CTA forms and stores its share of the chunk's
// rows); dX and the dA partials then run as the separate up-projection and weight-gradient launches.
// UR: rows of a unit, a 256-row chunk or (PC = false only) one 128-row tile, whose dB tree is then
// the unit's partial (the combine's first level adds the two tiles of each chunk). L: lanes that
// share one value of the dU rows step (4 where there are more than 8 slices, else 1). Both are
// compile-time so that the common case carries no registers for the others.
template <bool PC, int UR, int L>
__global__ void __launch_bounds__(BcCfg<PC>::kThreads, 1)
    bwd_cluster_kernel(const __grid_constant__ BcArgs args, uint32_t* status) {
  using C = BcCfg<PC>;
  constexpr int RP = C::RP;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + C::kArea);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto ready = [&](int s) { return bar0 + 8u * (C::kSlots + s); };
  auto empty = [&](int s) { return bar0 + 8u * (2 * C::kSlots + s); };
  auto tfull = [&](int t) { return bar0 + 8u * (3 * C::kSlots + t); };
  auto tempty = [&](int t) { return bar0 + 8u * (3 * C::kSlots + C::kTSlots + t); };
  auto duready = [&](int p) { return bar0 + 8u * (3 * C::kSlots + 2 * C::kTSlots + p); };
  const uint32_t duset = bar0 + 8u * (3 * C::kSlots + 2 * C::kTSlots + 2);
  const uint32_t drain = duset + 8u, never = duset + 16u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const uint32_t warp = warp_id(), lane = lane_id();
  const int CL = int(cluster_size()), rank = int(cluster_rank());
  const int cid = int(cluster_index()), ncl = int(cluster_count());
  const int M = args.M, K = args.K, N = args.N, S = args.S, n_ch = args.n_ch;
  static_assert((UR == kDyChunk || (!PC && UR == C::kBM)) && (L == 1 || L == 4), "unit shapes");
  const int n_kt = PC ? args.n_kt : 0;   // phase C column tiles (none without phase C)
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(full(s), 1);
      mbar_init(ready(s), C::kXfWarps);
      mbar_init(empty(s), 1);
    }
    for (int t = 0; t < C::kTSlots; ++t) {
      mbar_init(tfull(t), 1);
      mbar_init(tempty(t), C::kEpiWarps);
    }
    mbar_init(duready(0), CL);
    mbar_init(duready(1), CL);
    mbar_init(duset, 1);
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0u;
    mbar_fence_init();
    prefetch_map(&args.dy);
    prefetch_map(&args.b);
    prefetch_map(&args.u);
    if constexpr (PC) {
      prefetch_map(&args.x);
      prefetch_map(&args.a);
      prefetch_map(&args.dx);
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
  cluster_sync_all();          // every peer's mbarriers are initialised before any remote arrival
  // valid column tiles of a slice, row tiles (halves) of a chunk
  auto n_tiles = [&](int sl) { return (min(N - sl * kDySlice, kDySlice) + 127) / 128; };
  auto r_tiles = [&](int ch) { return (min(M - ch * UR, UR) + C::kBM - 1) / C::kBM; };
  if (threadIdx.x == 0 && cid < n_ch && rank < S) {
    // the first dY tiles of this CTA's first slice, into L2 while the predecessor drains
    const int nnt = n_tiles(rank), nrt = r_tiles(cid);
    for (int i = 0, n = 0; i < nnt && n < 4; ++i)
      for (int j = 0; j < nrt && n < 4; ++j, ++n)
        for (int q = 0; q < 4; ++q) tma_prefetch_l2(&args.dy, rank * kDySlice + i * 128 + 32 * q, cid * UR + j * C::kBM);
  }
  grid_dependency_wait();      // predecessor done: its outputs may be this kernel's inputs
  grid_dependents_launch();
  const Abort ab = make_abort(abort_flag, status);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      if (stall_requested(status, kKindDy)) stall_wait(never, ab, 39);   // test hooks: a wait that runs out
      const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_last();
      Ring r;
      uint32_t issued = 0, parities = 0;
      bool first_c = true;
      auto take = [&](int bytes) -> int {   // the next slot, once free; -1 when aborting
        const int s = int(r.idx);
        const bool ok = wait(empty(s), r.phase ^ 1u, ab, 81);
        if (ok) {
          mbar_expect_tx(full(s), uint32_t(bytes));
          issued |= 1u << s;
          parities = (parities & ~(1u << s)) | (r.phase << s);
        }
        return ok ? s : -1;
      };
      for (int ch = cid; ch < n_ch; ch += ncl) {
        const int nrt = r_tiles(ch);
        // phase A: dY tiles of this CTA's slices (column tiles outer, row tiles inner), with b and u rows
        for (int sl = rank; sl < S; sl += CL) {
          const int nnt = n_tiles(sl);
          for (int i = 0; i < nnt; ++i)
            for (int j = 0; j < nrt; ++j) {
              const int s = take(C::kSlotBytes);
              if (s >= 0) {
                const uint32_t st = base + s * C::kSlotBytes;
                const int n0 = sl * kDySlice + i * 128, m0 = ch * UR + j * C::kBM;
#pragma unroll
                for (int q = 0; q < 4; ++q) tma_load(st + q * C::kSlabBytes, &args.dy, full(s), n0 + 32 * q, m0, pol_stream);
                tma_load(st + C::kTileBytes, &args.b, full(s), 0, n0, pol_keep);
                tma_load(st + C::kTileBytes + C::kWBytes, &args.u, full(s), 0, m0, pol_keep);
              }
              r.next<C::kSlots>();
            }
        }
        // phase C: x tiles [128 rows][128 columns] and the a columns of this CTA's column tiles
        for (int kt = rank; kt < n_kt; kt += CL)
          for (int hh = 0; hh < nrt; ++hh) {
            if (first_c) {
              first_c = false;
              if (stall_requested(status, kKindWgrad)) stall_wait(never, ab, 29);
              if (stall_requested(status, kKindUp)) stall_wait(never, ab, 10);
            }
            const int s = take(C::kXBytes + C::kABytes);
            if (s >= 0) {
              const uint32_t st = base + s * C::kSlotBytes;
              const int k0 = kt * 128, m0 = ch * kDyChunk + hh * C::kBM;
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {   // 64-row halves: columns 0..63, then 64..127
                tma_load(st + h2 * 16384u, &args.x, full(s), k0, m0 + 64 * h2, pol_stream);
                tma_load(st + h2 * 16384u + 8192u, &args.x, full(s), k0 + 64, m0 + 64 * h2, pol_stream);
              }
              tma_load(st + C::kXBytes, &args.a, full(s), k0, 0, pol_keep);                  // a[0..RP)[k0 .. +63]
              tma_load(st + C::kXBytes + RP * 128, &args.a, full(s), k0 + 64, 0, pol_keep);  // a[0..RP)[k0+64 .. +127]
            }
            r.next<C::kSlots>();
          }
      }
      for (int s = 0; s < C::kSlots; ++s)
        if (issued & (1u << s)) wait_drain(full(s), (parities >> s) & 1u, ab, 82);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    // The whole warp follows the schedule; one elected lane issues. Descriptors
    // are built for slot 0 and advanced by the slot offset.
    constexpr uint32_t idesc_du = idesc_bf16(128, RP, 0, 1);    // dV K-major, b MN-major
    constexpr uint32_t idesc_db = idesc_bf16(128, RP, 1, 1);    // dV^T MN-major, u MN-major
    constexpr uint32_t idesc_da = idesc_bf16(128, RP, 1, 1);    // x^T MN-major, du MN-major
    constexpr uint32_t idesc_dx = idesc_bf16(128, 128, 0, 1);   // du K-major, a MN-major
    const uint32_t du0 = base + uint32_t(C::kDuOff);
    uint64_t a_du[C::kLeaves], b_du[C::kLeaves], a_db[C::kLeaves], b_db[C::kLeaves], a_da[C::kLeaves];
#pragma unroll
    for (int j = 0; j < C::kLeaves; ++j) {
      // dU leaf j: dV columns 16j..16j+15 -> slab j/2, K-major, 64-byte swizzle (8-row groups 512 B apart)
      a_du[j] = smem_desc(base + (j >> 1) * C::kSlabBytes + 32u * (j & 1), 16u, 512u, kLayoutSW64);
      // b rows 16j..16j+15 of [128 n][16 r]: MN-major, 32-byte swizzle (8-row groups 256 B apart)
      b_du[j] = smem_desc(base + C::kTileBytes + j * 512u, 256u, 256u, kLayoutSW32);
      // dB leaf j: dV rows 16j..16j+15 seen MN-major: 32-column atoms one slab apart, 8-row groups 512 B apart
      a_db[j] = smem_desc(base + j * 1024u, uint32_t(C::kSlabBytes), 512u, kLayoutSW64);
      b_db[j] = smem_desc(base + C::kTileBytes + C::kWBytes + j * 512u, 256u, 256u, kLayoutSW32);
      // dA leaf j: x rows 16j..16j+15 (64-row half j/4), transposed view: MN-major, 128-byte swizzle,
      // 64-column blocks 8 KB apart, 8-row groups 1 KB apart
      a_da[j] = smem_desc(base + (j >> 2) * 16384u + (j & 3) * 2048u, 8192u, 1024u, kLayoutSW128);
    }
    Ring r, t;
    int k = 0;
    auto issue = [&](bool phase_a, int hh) {
      bool ok = wait(ready(r.idx), r.phase, ab, 83);
      ok = __all_sync(0xffffffffu, ok && wait(tempty(t.idx), t.phase ^ 1u, ab, 84));
      if (ok) {
        tc_fence_after();
        const uint32_t off = r.idx * C::kSlotBytes;
        const uint32_t d = tmem + t.idx * C::kTCols;
        if (elect_one()) {   // one lane issues the step's MMAs back to back
          if (phase_a) {
#pragma unroll
            for (int j = 0; j < C::kLeaves; ++j)
              mma_bf16(d + j * RP, desc_advance(a_du[j], off), desc_advance(b_du[j], off), idesc_du, 0u);
#pragma unroll
            for (int j = 0; j < C::kLeaves; ++j)
              mma_bf16(d + (C::kLeaves + j) * RP, desc_advance(a_db[j], off), desc_advance(b_db[j], off), idesc_db, 0u);
          } else {
            // du rows of this half, MN-major for dA (r contiguous), K-major for dX; 32-byte swizzle
            const uint32_t g0 = du0 + uint32_t(hh) * (C::kBM * RP * 2);
#pragma unroll
            for (int j = 0; j < C::kLeaves; ++j)
              mma_bf16(d + j * RP, desc_advance(a_da[j], off), smem_desc(g0 + j * 512u, 256u, 256u, kLayoutSW32),
                       idesc_da, 0u);
            mma_bf16(d + 128u, smem_desc(g0, 16u, 256u, kLayoutSW32),
                     smem_desc(base + off + C::kXBytes, RP * 128u, 1024u, kLayoutSW128), idesc_dx, 0u);
          }
          mma_commit(empty(r.idx));
          mma_commit(tfull(t.idx));
        }
        __syncwarp();
      }
      r.next<C::kSlots>();
      t.next<C::kTSlots>();
    };
    for (int ch = cid; ch < n_ch; ch += ncl, ++k) {
      const int nrt = r_tiles(ch);
      for (int sl = rank; sl < S; sl += CL) {
        const int nst = n_tiles(sl) * nrt;
        for (int i = 0; i < nst; ++i) issue(true, 0);
      }
      if (rank < n_kt) {
        const bool okd = __all_sync(0xffffffffu, wait(duset, uint32_t(k) & 1u, ab, 85));   // the chunk's dU rows
        (void)okd;
        for (int kt = rank; kt < n_kt; kt += CL)
          for (int hh = 0; hh < nrt; ++hh) issue(false, hh);
      }
    }
    if (elect_one()) mma_commit(drain);
    __syncwarp();
    wait_drain(drain, 0u, ab, 86);
  } else if (warp < 2 + C::kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;                        // column half of R (dU, dB, dA); of the tile (dX)
    const int et = int(threadIdx.x) - 64;
    const uint32_t tq = tmem + (uint32_t(q * 32) << 16);
    const int tr = q * 32 + lane;                         // TMEM lane: row (dU, dX) or column (dB, dA)
    const uint32_t stg0 = base + uint32_t(C::kStgOff) + (warp - 2) * C::kStg * C::kStgBytes;
    uint8_t* stg_ptr = gbase + C::kStgOff + (warp - 2) * C::kStg * C::kStgBytes;
    uint8_t* dutile = gbase + C::kDuOff;
    const uint64_t pol_out = policy_evict_first();
    const int R = args.R, rows_per_rank = UR / CL;
    Ring t;
    int sidx = 0, k = 0;
    for (int ch = cid; ch < n_ch; ch += ncl, ++k) {
      const int nrt = r_tiles(ch);
      // ---- phase A: dU slice partials and dB chunk partials of this CTA's slices
      for (int sl = rank; sl < S; sl += CL) {
        const int nnt = n_tiles(sl);
        float du_stk[2][C::kSliceLevels > 0 ? C::kSliceLevels : 1][C::kCPT];   // per row tile: tree stack
        float db_first[C::kCPT];
        bool ok_all = true;
#pragma unroll
        for (int i = 0; i < C::kSliceTiles; ++i) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float dun[C::kCPT], dbn[C::kCPT];
            if (i < nnt && j < nrt) {
              const bool ok = __all_sync(0xffffffffu, wait(tfull(t.idx), t.phase, ab, 87));
              ok_all = ok_all && ok;
              tc_fence_after();
              const uint32_t ta = tq + t.idx * C::kTCols + h * C::kCPT;
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
              if (ok && lane == 0) mbar_arrive(tempty(t.idx));
              t.next<C::kTSlots>();
            } else {
#pragma unroll
              for (int c = 0; c < C::kCPT; ++c) dun[c] = dbn[c] = 0.0f;   // zero leaves: neutral in the tree
            }
            // dU of row tile j: canonical tree over the slice's column tiles
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
              const int row = ch * UR + j * C::kBM + tr;
              if (ok_all && j < nrt && row < M) {
                float4* dst = reinterpret_cast<float4*>(args.du_part + (size_t(sl) * M + row) * RP + h * C::kCPT);
                dst[0] = make_float4(dun[0], dun[1], dun[2], dun[3]);
                dst[1] = make_float4(dun[4], dun[5], dun[6], dun[7]);
              }
            }
            // dB of column tile i: the unit's row tiles (one: its tree is the partial; two: added)
            if (UR == C::kBM) {
              const int col = sl * kDySlice + i * 128 + tr;
              if (j == 0 && ok_all && i < nnt && col < N) {
                float* dst = args.db_part + (size_t(ch) * RP + h * C::kCPT) * N + col;
#pragma unroll
                for (int c = 0; c < C::kCPT; ++c) dst[size_t(c) * N] = dbn[c];
              }
            } else if (j == 0) {
#pragma unroll
              for (int c = 0; c < C::kCPT; ++c) db_first[c] = dbn[c];
            } else {
              const int col = sl * kDySlice + i * 128 + tr;
              if (ok_all && i < nnt && col < N) {
                float* dst = args.db_part + (size_t(ch) * RP + h * C::kCPT) * N + col;
#pragma unroll
                for (int c = 0; c < C::kCPT; ++c) dst[size_t(c) * N] = __fadd_rn(db_first[c], dbn[c]);
              }
            }
          }
        }
      }
      // ---- the cluster meets: every CTA's dU partials of the chunk are stored
      named_bar(1, 32 * C::kEpiWarps);
      if (et == 0)
        for (int p = 0; p < CL; ++p) mbar_arrive_peer(peer_addr(duready(k & 1), uint32_t(p)));
      const bool okx = __all_sync(0xffffffffu, wait_cluster(duready(k & 1), uint32_t(k >> 1) & 1u, ab, 88));
      // ---- dU rows of the chunk: canonical tree over the slices, BF16, into the swizzled tile
      // (32-byte rows: chunk ^ ((row / 4) % 2)); rank r stores its share of du
      // Without phase C a CTA forms its share only.
      // More than 8 slices: four consecutive lanes per value (the rows kernel's four-lane tree, the
      // same bits), all four active together (the conditions below are the same for the four).
      const int i0 = PC ? 0 : rank * rows_per_rank, ni = PC ? UR : rows_per_rank;
      const int l4 = et & (L - 1);
      const unsigned gmask = 0xFu << (lane & 28u);
      for (int it = et / L; it < ni * (RP / 8); it += 32 * C::kEpiWarps / L) {
        const int i = i0 + it / (RP / 8), gg = it % (RP / 8);
        const int row = ch * UR + i;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (okx && gg < R / 8 && row < M) {
          const float* pr = args.du_part + size_t(row) * RP + gg * 8;
          v = L == 4 ? slices_to_bf16x8_4lanes(pr, size_t(M) * RP, S, l4, gmask) : slices_to_bf16x8(pr, size_t(M) * RP, S);
          if (l4 == 0 && i / rows_per_rank == rank) *reinterpret_cast<uint4*>(args.du + size_t(row) * R + gg * 8) = v;
        }
        if constexpr (PC)
          if (l4 == 0) *reinterpret_cast<uint4*>(dutile + i * 32 + ((gg ^ ((i >> 2) & 1)) << 4)) = v;
      }
      fence_proxy_async();     // generic writes of the dU tile before the tensor core reads it
      named_bar(1, 32 * C::kEpiWarps);
      if (rank < n_kt && et == 0) mbar_arrive(duset);
      // ---- phase C: dA chunk partials and dX of this CTA's column tiles
      for (int kt = rank; kt < n_kt; kt += CL) {
        float da_first[C::kCPT];
        bool ok_all = true;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float dan[C::kCPT];
          if (hh < nrt) {
            const bool ok = __all_sync(0xffffffffu, wait(tfull(t.idx), t.phase, ab, 89));
            ok_all = ok_all && ok;
            tc_fence_after();
            const uint32_t ta = tq + t.idx * C::kTCols;
            float x0[8], x1[8];
            leaves4_tree(ta + h * C::kCPT, ok, x0);           // dA leaves 0..3 (rows 0..63 of the half)
            leaves4_tree(ta + h * C::kCPT + 4 * RP, ok, x1);  // dA leaves 4..7
#pragma unroll
            for (int c = 0; c < C::kCPT; ++c) dan[c] = __fadd_rn(x0[c], x1[c]);
            // dX rows hh * 128 + q * 32 + lane, columns kt * 128 + h * 64 .. + 63: two 32-column boxes
            const int row0 = ch * kDyChunk + hh * C::kBM + q * 32;
#pragma unroll
            for (int bx = 0; bx < 2; ++bx) {
              const int col0 = h * 64 + bx * 32;
              const int gcol = kt * 128 + col0;
              if (gcol >= K) break;                          // uniform over the warp
              if (lane == 0) tma_store_wait_read<C::kStg - 1>();   // this buffer's previous store has read it
              __syncwarp();
              uint32_t v[4][8];
#pragma unroll
              for (int b8 = 0; b8 < 4; ++b8)
#pragma unroll
                for (int e = 0; e < 8; ++e) v[b8][e] = 0u;
              if (ok) {
#pragma unroll
                for (int b8 = 0; b8 < 4; ++b8) tmem_ld8(ta + 128u + col0 + b8 * 8, v[b8]);
                tmem_ld_wait();
              }
#pragma unroll
              for (int b8 = 0; b8 < 4; ++b8) reg_fence(v[b8]);
              // 32 rows x 32 FP32 columns: 128-byte rows, 128-byte swizzle, chunk ^ (row % 8)
              uint8_t* buf = stg_ptr + sidx * C::kStgBytes;
#pragma unroll
              for (int cc = 0; cc < 8; ++cc)
                *reinterpret_cast<uint4*>(buf + lane * 128 + ((cc ^ (lane & 7)) * 16)) =
                    make_uint4(v[cc / 2][(cc % 2) * 4], v[cc / 2][(cc % 2) * 4 + 1], v[cc / 2][(cc % 2) * 4 + 2],
                               v[cc / 2][(cc % 2) * 4 + 3]);
              fence_proxy_async();
              __syncwarp();
              if (lane == 0) {
                if (ok && row0 < M) tma_store(&args.dx, stg0 + sidx * C::kStgBytes, gcol, row0, pol_out);
                tma_store_commit();   // one group per buffer use, empty or not
              }
              sidx = (sidx + 1) % C::kStg;
            }
            tc_fence_before();
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(tempty(t.idx));
            t.next<C::kTSlots>();
          } else {
#pragma unroll
            for (int c = 0; c < C::kCPT; ++c) dan[c] = 0.0f;   // zero leaves: neutral in the tree
          }
          if (hh == 0) {
#pragma unroll
            for (int c = 0; c < C::kCPT; ++c) da_first[c] = dan[c];
          } else {
            const int col = kt * 128 + tr;
            if (ok_all && col < K) {
              float* dst = args.da_part + (size_t(ch) * RP + h * C::kCPT) * K + col;
#pragma unroll
              for (int c = 0; c < C::kCPT; ++c) dst[size_t(c) * K] = __fadd_rn(da_first[c], dan[c]);
            }
          }
        }
      }
    }
    if (lane == 0) tma_store_wait_all<0>();
  } else {
    // ---------------------------------------------------- dV = bf16(dY*alpha)
    // Phase A slots are transformed in place; phase C slots are passed on once their copies landed,
    // so that `ready` marks every slot the MMA issuer may read.
    const int tt = int(threadIdx.x) - 32 * (2 + C::kEpiWarps);
    const float alpha = args.alpha;
    const uint32_t a2 = pow2_bf16x2(alpha);
    Ring r;
    auto pass = [&](bool transform) {
      if (wait(full(r.idx), r.phase, ab, 90)) {
        if (transform && !dv_is_dy(alpha)) {
          uint4* tile = reinterpret_cast<uint4*>(gbase + size_t(r.idx) * C::kSlotBytes);
#pragma unroll
          for (int e = 0; e < C::kTileBytes / 16 / (32 * C::kXfWarps); ++e)
            tile[tt + 32 * C::kXfWarps * e] = dv_bf16x8(tile[tt + 32 * C::kXfWarps * e], alpha, a2);
          fence_proxy_async();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(ready(r.idx));
      }
      r.next<C::kSlots>();
    };
    for (int ch = cid; ch < n_ch; ch += ncl) {
      const int nrt = r_tiles(ch);
      for (int sl = rank; sl < S; sl += CL) {
        const int nst = n_tiles(sl) * nrt;
        for (int i = 0; i < nst; ++i) pass(true);
      }
      for (int kt = rank; kt < n_kt; kt += CL)
        for (int hh = 0; hh < nrt; ++hh) pass(false);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();          // no CTA leaves while a peer may still arrive on its mbarriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool PC>
static cudaLaunchConfig_t bc_config(int cl, int ncl, cudaStream_t st, cudaLaunchAttribute (&attr)[2], int nattr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(ncl * cl));
  cfg.blockDim = dim3(BcCfg<PC>::kThreads);
  cfg.dynamicSmemBytes = BcCfg<PC>::kSmem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(cl);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = unsigned(nattr);
  return cfg;
}

template <bool PC, int UR, int L>
static cudaError_t bc_launch(BcArgs& a, uint32_t* status, int cl, int ncl, cudaStream_t st) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = bc_config<PC>(cl, ncl, st, attr, 2);
  return cudaLaunchKernelEx(&cfg, bwd_cluster_kernel<PC, UR, L>, a, status);
}

template <bool PC, int UR, int L>
static cudaError_t bc_prepare() {
  return cudaFuncSetAttribute(bwd_cluster_kernel<PC, UR, L>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(BcCfg<PC>::kSmem));
}

// every instance has the same threads, shared memory and one CTA per SM: one stands for all
cudaError_t bwd_cluster_max_clusters(bool phase_c, int cl, int* n) {
  cudaLaunchAttribute attr[2];
  if (phase_c) {
    cudaLaunchConfig_t cfg = bc_config<true>(cl, 1, nullptr, attr, 1);
    return cudaOccupancyMaxActiveClusters(n, bwd_cluster_kernel<true, kDyChunk, 1>, &cfg);
  }
  cudaLaunchConfig_t cfg = bc_config<false>(cl, 1, nullptr, attr, 1);
  return cudaOccupancyMaxActiveClusters(n, bwd_cluster_kernel<false, kDyChunk, 1>, &cfg);
}

cudaError_t launch_bwd_cluster(bool phase_c, BcArgs& a, uint32_t* status, int cl, int ncl, cudaStream_t st) {
  a.S = int(ceil_div(a.N, kDySlice));
  if (phase_c) a.unit_rows = kDyChunk;
  if (a.unit_rows != kDyChunk && a.unit_rows != 128) return cudaErrorInvalidValue;
  a.n_ch = int(ceil_div(a.M, a.unit_rows));
  a.n_kt = int(ceil_div(a.K, 128));
  if (cl < 1 || cl > 8 || (256 % cl) != 0 || ncl < 1) return cudaErrorInvalidValue;
  const bool many = a.S > 8;   // four lanes per value in the dU rows step
  if (phase_c)
    return many ? bc_launch<true, kDyChunk, 4>(a, status, cl, ncl, st) : bc_launch<true, kDyChunk, 1>(a, status, cl, ncl, st);
  if (a.unit_rows == kDyChunk)
    return many ? bc_launch<false, kDyChunk, 4>(a, status, cl, ncl, st) : bc_launch<false, kDyChunk, 1>(a, status, cl, ncl, st);
  return many ? bc_launch<false, 128, 4>(a, status, cl, ncl, st) : bc_launch<false, 128, 1>(a, status, cl, ncl, st);
}

cudaError_t prepare_bwd_cluster() {
  cudaError_t e;
  if ((e = bc_prepare<true, kDyChunk, 1>()) != cudaSuccess) return e;
  if ((e = bc_prepare<true, kDyChunk, 4>()) != cudaSuccess) return e;
  if ((e = bc_prepare<false, kDyChunk, 1>()) != cudaSuccess) return e;
  if ((e = bc_prepare<false, kDyChunk, 4>()) != cudaSuccess) return e;
  if ((e = bc_prepare<false, 128, 1>()) != cudaSuccess) return e;
  return bc_prepare<false, 128, 4>();
}

}  // namespace lora
