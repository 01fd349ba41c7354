// fwd_cluster.cu -- the forward pass in one launch of thread-block clusters:
//   U partials:  U[m][r] = sum_k x[m][k] * a[r][k] over K-slices   ("U = X @ A^T")
//   U rows:      U = bf16(canonical tree over the slices)          (rounded once, to BF16)
//   dY_lora:     dY_lora[m][n] = fp32(sum_r u[m][r] * b[n][r]) * alpha   ("(U @ B^T) * alpha")
// (page "[DSv4][P5-3] shared_grouped_lora_delta: CUDA + Triton, both
// batch-invariant", section "Summary"; its review thread asks for GEMM1 and
// GEMM2 in one kernel with U still stored, and for the alpha scale in the
// epilogue.)
//
// A cluster of CL CTAs (2, 4 or 8 SMs that the hardware runs together) owns one
// 128-row tile at a time; clusters take tiles round robin. CTA rank r of the
// cluster streams the K-slices r, r + CL, ... of the tile's X rows (one pass,
// TMA, 64-byte-swizzled 128 x 32 K-slabs), forms each slice's FP32 partial with
// the same 16-term tensor-core leaves and the same canonical tree as the
// standalone down-projection, and stores it in the workspace. Then the cluster
// meets: every CTA arrives on an mbarrier in each peer's shared memory (release
// at cluster scope) and waits on its own (acquire), reads all slice partials of
// the tile back from L2, adds them by the canonical tree over the slices,
// rounds to BF16 and writes the tile's U rows into its own shared memory (the
// A operand of the expansion, in the tensor core's swizzled layout); rank r
// also stores its 128 / CL rows of U. Each CTA then expands its column tiles
// r, r + CL, ... of dY_lora (the cluster writes neighbouring tiles at the same
// time), alpha and the TMA stores fused into the epilogue.
//
// The U rows are those of the rows kernel, and dY_lora that of the standalone
// up-projection, bit for bit: the same leaves, trees and rounding points; the
// cluster only changes which SM computes what. Peers wait for each other only
// inside a cluster, whose CTAs are resident together, so a plain (clustered)
// launch suffices; every wait is bounded.
//
// Warp roles: 0 = X / A producer (TMA), 1 = down MMA issuer (TMEM owner),
// 2..9 = epilogue (down leaves -> partials, the U rows, dY_lora stores),
// 10 = B producer, 11 = up MMA issuer. TMEM: columns [0, 256) hold the down
// leaf groups, [256, 512) two expansion buffers, so the down MMAs of the next
// tile run while the epilogue stores this one.
#include "common.cuh"
#include "kernels.h"

namespace lora {

template <int RP, bool UP>
struct FcCfg {
  static constexpr int kBM = 128, kBK = 64;
  // down-projection stages: X [128][64] as two [128][32] K-slabs + a [RP][64]
  static constexpr int kInBytes = kBM * kBK * 2;
  static constexpr int kSlabBytes = kInBytes / 2;
  static constexpr int kWBytes = RP * kBK * 2;
  static constexpr int kDStageBytes = kInBytes + kWBytes;
  static constexpr int kDStages = UP ? 6 : 10;           // without the expansion: a deeper read ring
  static constexpr int kLeaves = kBK / 16;               // leaves per stage
  static constexpr int kGroupCols = kLeaves * RP;        // TMEM columns per stage
  static constexpr int kGroups = 256 / kGroupCols;       // down TMEM ring in columns [0, 256)
  static constexpr int kSlice = down_slice(RP);
  static constexpr int kGS = kSlice / kBK;               // stages per slice
  static constexpr int kLevels = kGS == 16 ? 4 : (kGS == 8 ? 3 : (kGS == 4 ? 2 : (kGS == 2 ? 1 : 0)));
  static constexpr int kCPT = RP / 2;                    // down epilogue: columns per thread
  static constexpr int kCH = kCPT < 16 ? kCPT : 16;
  // expansion: units of 128 rows x kBN columns, one leaf per 16 of RP
  static constexpr int kUpLeaves = RP / 16;
  static constexpr int kBufCols = 128, kBufs = 2;        // TMEM columns [256, 512)
  static constexpr int kBN = kBufCols / kUpLeaves;
  static constexpr int kSpan = RP * 2;                   // bytes of a U / b row
  static constexpr int kUBytes = kBM * RP * 2;
  static constexpr int kBBytes = kBN * RP * 2;
  static constexpr int kBStages = 4;
  static constexpr int kHalfCols = kBN / 2;              // columns per epilogue warp and unit
  static constexpr int kBoxes = kHalfCols / 32;          // 32-column store boxes per warp and unit
  static constexpr int kStg = 2, kStgBytes = 32 * 32 * 4;
  static constexpr int kEpiWarps = 8;
  static constexpr int kThreads = 32 * 12;
  // shared memory, from the 1024-byte aligned base
  static constexpr size_t kUOff = size_t(kDStages) * kDStageBytes;
  static constexpr size_t kBOff = kUOff + kUBytes;
  static constexpr size_t kStgOff = kBOff + size_t(kBStages) * kBBytes;
  static constexpr size_t kArea = UP ? kStgOff + size_t(kEpiWarps) * kStg * kStgBytes : kUOff;
  // mbarriers: down ring (full, empty), down TMEM (full, empty), b ring (full, empty),
  // up TMEM (full, empty), U exchange [2], U tile set, drains (down, up), never
  static constexpr int kB0 = 0, kB1 = kB0 + 2 * kDStages, kB2 = kB1 + 2 * kGroups, kB3 = kB2 + 2 * kBStages,
                       kB4 = kB3 + 2 * kBufs;
  static constexpr int kNumBars = kB4 + 6;
  static constexpr size_t kSmem = kArea + 1024 + kNumBars * 8 + 16;
  static_assert(kDStageBytes % 1024 == 0 && kUOff % 1024 == 0 && kStgOff % 1024 == 0, "1024-byte aligned tiles");
  static_assert((1 << kLevels) == kGS && kGroups >= 2 && kBoxes >= 1, "tree and ring shapes");
  static_assert(kSmem < 227 * 1024, "one CTA per SM");
};

// 16-byte chunk g of row i of a [128][RP] BF16 tile in the tensor core's swizzled K-major layout
// (swizzle span = one row of 2 RP bytes; the tile starts 1024-byte aligned): the chunk index is
// XORed with address bits 7.. of the row, as a TMA load with that swizzle mode would place it.
template <int RP>
__device__ __forceinline__ uint32_t utile_offset(int i, int g) {
  if constexpr (RP == 16) return uint32_t(i * 32 + ((g ^ ((i >> 2) & 1)) << 4));
  else if constexpr (RP == 32) return uint32_t(i * 64 + ((g ^ ((i >> 1) & 3)) << 4));
  else return uint32_t(i * 128 + ((g ^ (i & 7)) << 4));
}

// UP = false: the down-projection and the U rows only (each CTA forms and stores its share of the
// tile's rows); the expansion then runs as the separate up-projection launch.
template <int RP, bool YBF, bool UP>
__global__ void __launch_bounds__(FcCfg<RP, UP>::kThreads, 1)
    fwd_cluster_kernel(const __grid_constant__ FcArgs args, uint32_t* status) {
  using C = FcCfg<RP, UP>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + C::kArea);
  const uint32_t bar0 = smem_u32(bars);
  auto dfull = [&](int s) { return bar0 + 8u * (C::kB0 + s); };
  auto dempty = [&](int s) { return bar0 + 8u * (C::kB0 + C::kDStages + s); };
  auto tfull = [&](int g) { return bar0 + 8u * (C::kB1 + g); };
  auto tempty = [&](int g) { return bar0 + 8u * (C::kB1 + C::kGroups + g); };
  auto bfull = [&](int s) { return bar0 + 8u * (C::kB2 + s); };
  auto bempty = [&](int s) { return bar0 + 8u * (C::kB2 + C::kBStages + s); };
  auto ufull = [&](int b) { return bar0 + 8u * (C::kB3 + b); };
  auto uempty = [&](int b) { return bar0 + 8u * (C::kB3 + C::kBufs + b); };
  auto uready = [&](int p) { return bar0 + 8u * (C::kB4 + p); };   // the cluster's partials of a tile stored
  const uint32_t uset = bar0 + 8u * (C::kB4 + 2);                    // the U tile is in shared memory
  const uint32_t drain_d = bar0 + 8u * (C::kB4 + 3), drain_u = drain_d + 8u;
  const uint32_t never = drain_d + 16u;                              // completed by nothing (stall hook)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const uint32_t warp = warp_id(), lane = lane_id();
  const int CL = int(cluster_size()), rank = int(cluster_rank());
  const int cid = int(cluster_index()), ncl = int(cluster_count());
  const int M = args.M, K = args.K, N = args.N, S = args.S, n_mt = args.n_mt;
  // column tiles of the expansion: none without it (its shared memory is then not allocated)
  const int n_nt = UP ? args.n_nt : 0;
  const bool has_up = rank < n_nt;   // this CTA expands some column tile of every row tile
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kDStages; ++s) {
      mbar_init(dfull(s), 1);
      mbar_init(dempty(s), 1);
    }
    for (int g = 0; g < C::kGroups; ++g) {
      mbar_init(tfull(g), 1);
      mbar_init(tempty(g), C::kEpiWarps);
    }
    for (int s = 0; s < C::kBStages; ++s) {
      mbar_init(bfull(s), 1);
      mbar_init(bempty(s), 1);
    }
    for (int b = 0; b < C::kBufs; ++b) {
      mbar_init(ufull(b), 1);
      mbar_init(uempty(b), C::kEpiWarps);
    }
    mbar_init(uready(0), CL);
    mbar_init(uready(1), CL);
    mbar_init(uset, 1);
    mbar_init(drain_d, 1);
    mbar_init(drain_u, 1);
    mbar_init(never, 1);
    *abort_flag = 0u;
    mbar_fence_init();
    prefetch_map(&args.x);
    prefetch_map(&args.a);
    if constexpr (UP) {
      prefetch_map(&args.b);
      prefetch_map(&args.out);
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
  if (threadIdx.x == 0 && cid < n_mt && rank < S) {
    // the first X tiles of this CTA's first slice, into L2 while the predecessor drains
    const int nkb = (min(K - rank * C::kSlice, C::kSlice) + C::kBK - 1) / C::kBK;
    for (int kb = 0; kb < min(nkb, 8); ++kb) {
      tma_prefetch_l2(&args.x, rank * C::kSlice + kb * C::kBK, cid * C::kBM);
      tma_prefetch_l2(&args.x, rank * C::kSlice + kb * C::kBK + 32, cid * C::kBM);
    }
  }
  grid_dependency_wait();      // predecessor done: its outputs may be this kernel's inputs
  grid_dependents_launch();
  const Abort ab = make_abort(abort_flag, status);
  auto nkb_of = [&](int sl) { return (min(K - sl * C::kSlice, C::kSlice) + C::kBK - 1) / C::kBK; };

  if (warp == 0) {
    // ----------------------------------------------------- X / A producer
    if (lane == 0) {
      if (stall_requested(status, kKindDown)) stall_wait(never, ab, 9);   // test hook: a wait that runs out
      const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_last();
      Ring r;
      uint32_t issued = 0, parities = 0;
      for (int mt = cid; mt < n_mt; mt += ncl)
        for (int sl = rank; sl < S; sl += CL) {
          const int nkb = nkb_of(sl);
          for (int kb = 0; kb < nkb; ++kb) {
            if (wait(dempty(r.idx), r.phase ^ 1u, ab, 61)) {
              const uint32_t st = base + r.idx * C::kDStageBytes;
              const int k = sl * C::kSlice + kb * C::kBK;
              mbar_expect_tx(dfull(r.idx), C::kDStageBytes);
              tma_load(st, &args.x, dfull(r.idx), k, mt * C::kBM, pol_stream);
              tma_load(st + C::kSlabBytes, &args.x, dfull(r.idx), k + 32, mt * C::kBM, pol_stream);
              tma_load(st + C::kInBytes, &args.a, dfull(r.idx), k, 0, pol_keep);
              issued |= 1u << r.idx;
              parities = (parities & ~(1u << r.idx)) | (r.phase << r.idx);
            }
            r.next<C::kDStages>();
          }
        }
      for (int s = 0; s < C::kDStages; ++s)
        if (issued & (1u << s)) wait_drain(dfull(s), (parities >> s) & 1u, ab, 62);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ down MMA issuer
    constexpr uint32_t idesc = idesc_bf16(128, RP, 0, 0);
    uint64_t adesc[C::kLeaves], wdesc[C::kLeaves];
#pragma unroll
    for (int j = 0; j < C::kLeaves; ++j) {
      // X slab j/2: K-major, 64-byte rows, 64-byte swizzle, 8-row groups 512 bytes apart
      adesc[j] = smem_desc(base + (j >> 1) * C::kSlabBytes + 32u * (j & 1), 16u, 512u, kLayoutSW64);
      // a tile [RP][64 k]: K-major, 128-byte swizzle
      wdesc[j] = smem_desc(base + C::kInBytes + 32u * j, 16u, 1024u, kLayoutSW128);
    }
    Ring r, g;
    for (int mt = cid; mt < n_mt; mt += ncl)
      for (int sl = rank; sl < S; sl += CL) {
        const int nkb = nkb_of(sl);
        for (int kb = 0; kb < nkb; ++kb) {
          bool ok = wait(dfull(r.idx), r.phase, ab, 63);
          ok = __all_sync(0xffffffffu, ok && wait(tempty(g.idx), g.phase ^ 1u, ab, 64));
          if (ok) {
            tc_fence_after();
            const uint32_t off = r.idx * C::kDStageBytes;
            const uint32_t d = tmem + g.idx * C::kGroupCols;
            if (elect_one()) {   // one lane issues the stage's MMAs back to back
#pragma unroll
              for (int j = 0; j < C::kLeaves; ++j)   // fresh accumulator: one leaf
                mma_bf16(d + j * RP, desc_advance(adesc[j], off), desc_advance(wdesc[j], off), idesc, 0u);
              mma_commit(dempty(r.idx));
              mma_commit(tfull(g.idx));
            }
            __syncwarp();
          }
          r.next<C::kDStages>();
          g.next<C::kGroups>();
        }
      }
    if (elect_one()) mma_commit(drain_d);
    __syncwarp();
    wait_drain(drain_d, 0u, ab, 65);
  } else if (warp < 2 + C::kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                  // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;           // column half
    const int et = int(threadIdx.x) - 64;    // 0 .. 255
    const uint32_t tq = tmem + (uint32_t(q * 32) << 16);
    const uint32_t stg0 = base + uint32_t(C::kStgOff) + (warp - 2) * C::kStg * C::kStgBytes;
    uint8_t* stg_ptr = gbase + C::kStgOff + (warp - 2) * C::kStg * C::kStgBytes;
    uint8_t* utile = gbase + C::kUOff;
    const uint64_t pol_out = policy_evict_first();
    const float alpha = args.alpha;
    const int R = args.R, rows_per_rank = C::kBM / CL;
    Ring g, b;
    int sidx = 0, k = 0;
    for (int mt = cid; mt < n_mt; mt += ncl, ++k) {
      // (1) the slice partials of this CTA's slices of the tile
      for (int sl = rank; sl < S; sl += CL) {
        const int nkb = nkb_of(sl);
        const uint32_t tbase = tq + h * C::kCPT;
        float stack[C::kLevels > 0 ? C::kLevels : 1][C::kCPT];
        float node[C::kCPT];
        bool ok_all = true;
#pragma unroll
        for (int i = 0; i < C::kGS; ++i) {
          if (i < nkb) {
            const bool ok = __all_sync(0xffffffffu, wait(tfull(g.idx), g.phase, ab, 66));
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
          // canonical pairwise tree over the slice's stages: merge once per trailing one of i
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
        const int row = mt * C::kBM + q * 32 + lane;
        if (ok_all && row < M) {
          float4* dst = reinterpret_cast<float4*>(args.part + (size_t(sl) * M + row) * RP + h * C::kCPT);
#pragma unroll
          for (int c = 0; c < C::kCPT; c += 4) dst[c / 4] = make_float4(node[c], node[c + 1], node[c + 2], node[c + 3]);
        }
      }
      // (2) the cluster meets: every CTA's partials of the tile are stored (CTA barrier, then a
      // release at cluster scope on each peer's mbarrier); wait for all CL arrivals (acquire)
      named_bar(1, 32 * C::kEpiWarps);
      if (et == 0)
        for (int p = 0; p < CL; ++p) mbar_arrive_peer(peer_addr(uready(k & 1), uint32_t(p)));
      const bool okx = __all_sync(0xffffffffu, wait_cluster(uready(k & 1), uint32_t(k >> 1) & 1u, ab, 67));
      // (3) the U rows of the tile: canonical tree over the slices, BF16, into the swizzled U
      // tile (padded columns and rows past M are zero); rank r also stores its share of u.
      // Without the expansion a CTA forms its share only.
      // More than 8 slices: four consecutive lanes per value (the rows kernel's four-lane tree, the
      // same bits), all four active together (the conditions below are the same for the four).
      const int i0 = UP ? 0 : rank * rows_per_rank, ni = UP ? C::kBM : rows_per_rank;
      const int L = S > 8 ? 4 : 1, l4 = et & (L - 1);
      const unsigned gmask = 0xFu << (lane & 28u);
      for (int it = et / L; it < ni * (RP / 8); it += 32 * C::kEpiWarps / L) {
        const int i = i0 + it / (RP / 8), gg = it % (RP / 8);
        const int row = mt * C::kBM + i;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (okx && gg < R / 8 && row < M) {
          const float* pr = args.part + size_t(row) * RP + gg * 8;
          v = L == 4 ? slices_to_bf16x8_4lanes(pr, size_t(M) * RP, S, l4, gmask) : slices_to_bf16x8(pr, size_t(M) * RP, S);
          if (l4 == 0 && i / rows_per_rank == rank) *reinterpret_cast<uint4*>(args.u + size_t(row) * R + gg * 8) = v;
        }
        if constexpr (UP)
          if (l4 == 0) *reinterpret_cast<uint4*>(utile + utile_offset<RP>(i, gg)) = v;
      }
      fence_proxy_async();     // generic writes of the U tile before the tensor core reads it
      named_bar(1, 32 * C::kEpiWarps);
      if (has_up && et == 0) mbar_arrive(uset);
      // (4) dY_lora of this CTA's column tiles of the row tile
      for (int nt = rank; nt < n_nt; nt += CL) {
        const bool ok = __all_sync(0xffffffffu, wait(ufull(b.idx), b.phase, ab, 68));
        tc_fence_after();
        const int row0 = mt * C::kBM + q * 32;
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx) {
          const int col0 = h * C::kHalfCols + bx * 32;    // within the unit
          const int gcol = nt * C::kBN + col0;
          if (gcol >= N) break;                            // uniform over the warp
          if (lane == 0) tma_store_wait_read<C::kStg - 1>();   // this buffer's previous store has read it
          __syncwarp();
          uint32_t v[C::kUpLeaves][4][8];
#pragma unroll
          for (int j = 0; j < C::kUpLeaves; ++j)
#pragma unroll
            for (int b8 = 0; b8 < 4; ++b8)
#pragma unroll
              for (int e = 0; e < 8; ++e) v[j][b8][e] = 0u;
          if (ok) {
#pragma unroll
            for (int j = 0; j < C::kUpLeaves; ++j)
#pragma unroll
              for (int b8 = 0; b8 < 4; ++b8)
                tmem_ld8(tq + 256u + b.idx * C::kBufCols + j * C::kBN + col0 + b8 * 8, v[j][b8]);
            tmem_ld_wait();
          }
#pragma unroll
          for (int j = 0; j < C::kUpLeaves; ++j)
#pragma unroll
            for (int b8 = 0; b8 < 4; ++b8) reg_fence(v[j][b8]);
          // leaf tree of column e (one or two leaves) and the alpha multiply
          auto value = [&](int e) {
            const int b8 = e / 8, c = e % 8;
            float s = __uint_as_float(v[0][b8][c]);
            if constexpr (C::kUpLeaves == 2) s = __fadd_rn(s, __uint_as_float(v[1][b8][c]));
            return __fmul_rn(s, alpha);
          };
          uint8_t* buf = stg_ptr + sidx * C::kStgBytes;
          if constexpr (YBF) {
            // 32 rows x 32 BF16 columns: 64-byte rows, 64-byte swizzle, chunk ^ ((row / 2) % 4)
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              float f[8];
#pragma unroll
              for (int t8 = 0; t8 < 8; ++t8) f[t8] = value(cc * 8 + t8);
              *reinterpret_cast<uint4*>(buf + lane * 64 + ((cc ^ ((lane >> 1) & 3)) * 16)) = pack_bf16x8(f);
            }
          } else {
            // 32 rows x 32 FP32 columns: 128-byte rows, 128-byte swizzle, chunk ^ (row % 8)
#pragma unroll
            for (int cc = 0; cc < 8; ++cc)
              *reinterpret_cast<float4*>(buf + lane * 128 + ((cc ^ (lane & 7)) * 16)) =
                  make_float4(value(cc * 4), value(cc * 4 + 1), value(cc * 4 + 2), value(cc * 4 + 3));
          }
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) {
            if (ok && row0 < M) tma_store(&args.out, stg0 + sidx * C::kStgBytes, gcol, row0, pol_out);
            tma_store_commit();   // one group per buffer use, empty or not
          }
          sidx = (sidx + 1) % C::kStg;
        }
        tc_fence_before();
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(uempty(b.idx));
        b.next<C::kBufs>();
      }
    }
    if (lane == 0) tma_store_wait_all<0>();
  } else if (warp == 10) {
    // ----------------------------------------------------------- b producer
    if (lane == 0 && has_up) {
      if (stall_requested(status, kKindUp)) stall_wait(never, ab, 10);   // test hook: a wait that runs out
      const uint64_t pol = policy_evict_last();
      Ring r;
      uint32_t issued = 0, parities = 0;
      for (int mt = cid; mt < n_mt; mt += ncl)
        for (int nt = rank; nt < n_nt; nt += CL) {
          if (wait(bempty(r.idx), r.phase ^ 1u, ab, 69)) {
            const uint32_t st = base + uint32_t(C::kBOff) + r.idx * C::kBBytes;
            mbar_expect_tx(bfull(r.idx), C::kBBytes);
            tma_load(st, &args.b, bfull(r.idx), 0, nt * C::kBN, pol);   // b rows n .. n + kBN
            issued |= 1u << r.idx;
            parities = (parities & ~(1u << r.idx)) | (r.phase << r.idx);
          }
          r.next<C::kBStages>();
        }
      for (int s = 0; s < C::kBStages; ++s)
        if (issued & (1u << s)) wait_drain(bfull(s), (parities >> s) & 1u, ab, 70);
    }
  } else {
    // -------------------------------------------------------- up MMA issuer
    if (lane == 0 && has_up) {
      constexpr uint32_t idesc = idesc_bf16(128, C::kBN, 0, 0);
      constexpr uint32_t lay = layout_for_span(C::kSpan);
      Ring r, b;
      int k = 0;
      for (int mt = cid; mt < n_mt; mt += ncl, ++k) {
        const bool oku = wait(uset, uint32_t(k) & 1u, ab, 71);   // the tile's U rows are in shared memory
        for (int nt = rank; nt < n_nt; nt += CL) {
          bool ok = oku && wait(bfull(r.idx), r.phase, ab, 72);
          ok = ok && wait(uempty(b.idx), b.phase ^ 1u, ab, 73);
          if (ok) {
            tc_fence_after();
            const uint32_t st = base + uint32_t(C::kBOff) + r.idx * C::kBBytes;
#pragma unroll
            for (int j = 0; j < C::kUpLeaves; ++j) {
              // U tile and b tile: K-major, rows of 2 RP bytes, swizzle span = row; K step j = +32 bytes
              const uint64_t adesc = smem_desc(base + uint32_t(C::kUOff) + 32u * j, 16u, 8u * C::kSpan, lay);
              const uint64_t bdesc = smem_desc(st + 32u * j, 16u, 8u * C::kSpan, lay);
              mma_bf16(tmem + 256u + b.idx * C::kBufCols + j * C::kBN, adesc, bdesc, idesc, 0u);
            }
            mma_commit(bempty(r.idx));
            mma_commit(ufull(b.idx));
          }
          r.next<C::kBStages>();
          b.next<C::kBufs>();
        }
      }
      mma_commit(drain_u);
      wait_drain(drain_u, 0u, ab, 74);
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

template <int RP, bool YBF, bool UP>
static cudaError_t launch_inst(const FcArgs& a, uint32_t* status, int cl, int ncl, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(ncl * cl));
  cfg.blockDim = dim3(FcCfg<RP, UP>::kThreads);
  cfg.dynamicSmemBytes = FcCfg<RP, UP>::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(cl);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, fwd_cluster_kernel<RP, YBF, UP>, a, status);
}

template <int RP, bool YBF, bool UP>
static cudaError_t max_clusters_inst(int cl, int* n) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(cl));
  cfg.blockDim = dim3(FcCfg<RP, UP>::kThreads);
  cfg.dynamicSmemBytes = FcCfg<RP, UP>::kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(cl);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(n, fwd_cluster_kernel<RP, YBF, UP>, &cfg);
}

// Instance code: padded rank, BF16 output, expansion in the launch.
// (The output type matters only with the expansion.)
static int fc_code(int RP, bool y_bf16, bool up) { return RP * 4 + (y_bf16 && up ? 1 : 0) + (up ? 2 : 0); }

cudaError_t fwd_cluster_max_clusters(int RP, bool y_bf16, bool up, int cl, int* n) {
  switch (fc_code(RP, y_bf16, up)) {
    case 66: return max_clusters_inst<16, false, true>(cl, n);
    case 67: return max_clusters_inst<16, true, true>(cl, n);
    case 130: return max_clusters_inst<32, false, true>(cl, n);
    case 131: return max_clusters_inst<32, true, true>(cl, n);
    case 64: return max_clusters_inst<16, false, false>(cl, n);
    case 128: return max_clusters_inst<32, false, false>(cl, n);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fwd_cluster(int RP, bool y_bf16, bool up, FcArgs& a, uint32_t* status, int cl, int ncl,
                               cudaStream_t st) {
  a.S = int(ceil_div(a.K, down_slice(RP)));
  a.n_mt = int(ceil_div(a.M, 128));
  a.n_nt = int(ceil_div(a.N, fc_bn(RP)));
  if (cl < 1 || cl > 8 || (128 % cl) != 0 || ncl < 1) return cudaErrorInvalidValue;
  switch (fc_code(RP, y_bf16, up)) {
    case 66: return launch_inst<16, false, true>(a, status, cl, ncl, st);
    case 67: return launch_inst<16, true, true>(a, status, cl, ncl, st);
    case 130: return launch_inst<32, false, true>(a, status, cl, ncl, st);
    case 131: return launch_inst<32, true, true>(a, status, cl, ncl, st);
    case 64: return launch_inst<16, false, false>(a, status, cl, ncl, st);
    case 128: return launch_inst<32, false, false>(a, status, cl, ncl, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int RP, bool YBF, bool UP>
static cudaError_t prep_one() {
  return cudaFuncSetAttribute(fwd_cluster_kernel<RP, YBF, UP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(FcCfg<RP, UP>::kSmem));
}

cudaError_t prepare_fwd_cluster() {
  cudaError_t e;
  if ((e = prep_one<16, false, true>()) != cudaSuccess) return e;
  if ((e = prep_one<16, true, true>()) != cudaSuccess) return e;
  if ((e = prep_one<32, false, true>()) != cudaSuccess) return e;
  if ((e = prep_one<32, true, true>()) != cudaSuccess) return e;
  if ((e = prep_one<16, false, false>()) != cudaSuccess) return e;
  return prep_one<32, false, false>();
}

}  // namespace lora
