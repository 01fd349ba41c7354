// down_phase.cuh -- the reductions over the long dimension, as a kernel phase:
//   U  partials: U[m][r]  = sum_k x[m][k] * a[r][k]      (forward "U = X @ A^T")
//   dU partials: dU[m][r] = sum_n dv[m][n] * b[n][r],   dv = bf16(dy * alpha)
// (page "[DSv4][P5-3] shared_grouped_lora_delta: CUDA + Triton, both
// batch-invariant", section "Summary"; dV is formed in shared memory and never
// stored, rounding point "D4").
//
// Work unit = (128-row tile, slice of the reduction dimension); units are
// numbered row-tile major (u0 + mt * n_sl + sl), so with units taken in order
// the row tiles complete one after another. A persistent CTA streams the
// unit's 128 x 64 BF16 input tiles through a TMA/mbarrier ring (one pass over
// the input; each tile lands as two 128 x 32 K-slabs with a 64-byte swizzle:
// measured on GB300, the tensor core reads this layout far faster than a
// 128-byte-swizzled 128 x 64 tile, whose MMA operand fetch otherwise adds ~40
// cycles per MMA to the streaming time), issues four tcgen05 MMAs (M=128,
// N=RP, K=16) per tile, each into its own fresh TMEM accumulator (a "leaf" =
// one 16-term dot product), and eight epilogue warps add the leaves with the
// canonical pairwise tree in FP32 (round to nearest). The unit's result is one
// FP32 partial per (row, r); the rows kernel (or the fused forward's rows
// step) finishes the same tree across slices and rounds to BF16.
//
// Warp roles: 0 = TMA producer, 1 = MMA issuer (and TMEM owner),
// 2..9 = epilogue (two warps per TMEM lane quarter, half of the columns each),
// 10..13 = dV transform (dU only).
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "sched.cuh"

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
  static constexpr int kWarps = 2 + kEpiWarps + kXfWarps;
  static constexpr int kCPT = RP / 2;                 // columns per epilogue thread
  static constexpr int kCH = kCPT < 16 ? kCPT : 16;   // columns per TMEM load batch
  static constexpr int kWSpan = DV ? RP * 2 : 128;    // swizzle span of the weight tile
  static constexpr int kPrefetch = 8;                 // input tiles warmed in L2 before the dependency wait
  static constexpr size_t kStageArea = size_t(kStages) * kStageBytes;   // from the 1024-byte aligned base
  static constexpr int kNumBars = 3 * kStages + 2 * kGroups + 2;        // ring, TMEM ring, drain, never
  static_assert((1 << kLevels) == kGS, "slice must hold a power-of-two number of tiles");
  static_assert(kGroups >= 2, "TMEM ring too shallow");
};

// The phase: GR = several sites in the table (otherwise one, read at fixed offsets).
template <int RP, bool DV, bool GR>
struct DownPhase {
  using C = DownCfg<RP, DV>;
  using Args = Sites<DownSite, GR ? kMaxSites : 1>;

  struct Bars {
    uint32_t b0;
    __device__ __forceinline__ uint32_t full(int s) const { return b0 + 8u * s; }
    __device__ __forceinline__ uint32_t ready(int s) const { return b0 + 8u * (C::kStages + s); }
    __device__ __forceinline__ uint32_t empty(int s) const { return b0 + 8u * (2 * C::kStages + s); }
    __device__ __forceinline__ uint32_t tfull(int g) const { return b0 + 8u * (3 * C::kStages + g); }
    __device__ __forceinline__ uint32_t tempty(int g) const { return b0 + 8u * (3 * C::kStages + C::kGroups + g); }
    __device__ __forceinline__ uint32_t drain() const { return b0 + 8u * (3 * C::kStages + 2 * C::kGroups); }
    __device__ __forceinline__ uint32_t never() const { return drain() + 8u; }   // completed by nothing
  };

  // site of unit u (sites are few and ordered by first unit)
  static __device__ __forceinline__ const DownSite& site(const Args& args, int u) {
    if constexpr (!GR) return args.s[0];
    int i = 0;
    while (i + 1 < args.n && u >= args.s[i + 1].u0) ++i;
    return args.s[i];
  }
  struct Unit {
    int mt, sl, k0, nkb;
  };
  static __device__ __forceinline__ Unit unit(const DownSite& S, int u) {
    const int lu = u - S.u0;
    Unit t;
    t.mt = lu / S.n_sl;
    t.sl = lu % S.n_sl;
    t.k0 = t.sl * C::kSlice;
    t.nkb = (min(S.Kred - t.k0, C::kSlice) + C::kBK - 1) / C::kBK;
    return t;
  }

  // thread 0, before the kernel's mbarrier init fence
  static __device__ void init(const Bars& B, const Args& args) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(B.full(s), 1);
      mbar_init(B.ready(s), C::kXfWarps > 0 ? C::kXfWarps : 1);
      mbar_init(B.empty(s), 1);
    }
    for (int g = 0; g < C::kGroups; ++g) {
      mbar_init(B.tfull(g), 1);
      mbar_init(B.tempty(g), C::kEpiWarps);
    }
    mbar_init(B.drain(), 1);
    mbar_init(B.never(), 1);
    for (int i = 0; i < (GR ? args.n : 1); ++i) {
      prefetch_map(&args.s[i].in);
      prefetch_map(&args.s[i].w);
    }
  }
  // thread 0: the first input tiles of unit u into L2 (before the grid dependency wait)
  static __device__ void warm_l2(const Args& args, int u) {
    if (u < 0 || u >= args.total) return;
    const DownSite& S = site(args, u);
    const Unit t = unit(S, u);
    for (int kb = 0; kb < min(t.nkb, C::kPrefetch); ++kb) {
      tma_prefetch_l2(&S.in, t.k0 + kb * C::kBK, t.mt * C::kBM);
      tma_prefetch_l2(&S.in, t.k0 + kb * C::kBK + 32, t.mt * C::kBM);
    }
  }

  // All warps of the phase call this (warps beyond kWarps return at once). `base`: 1024-byte
  // aligned start of the stage area (generic pointer gbase). PS / RS: the producer's and the
  // other roles' unit sequences; hook.stored(k): an epilogue warp has stored the partial of its
  // k-th unit (0, 1, ...). Returns when every copy and MMA the phase issued has completed.
  template <class PS, class RS, class Hook>
  static __device__ void run(const Args& args, uint8_t* gbase, uint32_t base, const Bars& B, uint32_t tmem,
                             const Abort& ab, const uint32_t* status, PS ps, RS rs, Hook& hook) {
    const uint32_t warp = warp_id(), lane = lane_id();
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        if (stall_requested(status, kKindDown)) stall_wait(B.never(), ab, 9);   // test hook: a wait that runs out
        const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_last();
        Ring r;
        uint32_t issued = 0, parities = 0;
        for (int u = ps.first(); u >= 0; u = ps.next(u)) {
          const DownSite& S = site(args, u);
          const Unit t = unit(S, u);
          for (int kb = 0; kb < t.nkb; ++kb) {
            if (wait(B.empty(r.idx), r.phase ^ 1u, ab, 1)) {
              const uint32_t st = base + r.idx * C::kStageBytes;
              const int k = t.k0 + kb * C::kBK;
              mbar_expect_tx(B.full(r.idx), C::kStageBytes);
              tma_load(st, &S.in, B.full(r.idx), k, t.mt * C::kBM, pol_stream);                     // k .. k+31
              tma_load(st + C::kSlabBytes, &S.in, B.full(r.idx), k + 32, t.mt * C::kBM, pol_stream);  // k+32 .. k+63
              if (DV) tma_load(st + C::kInBytes, &S.w, B.full(r.idx), 0, k, pol_keep);   // b[n][r], n = k..k+63
              else tma_load(st + C::kInBytes, &S.w, B.full(r.idx), k, 0, pol_keep);      // a[r][k..k+63]
              issued |= 1u << r.idx;
              parities = (parities & ~(1u << r.idx)) | (r.phase << r.idx);
            }
            r.next<C::kStages>();
          }
        }
        // never leave with a copy in flight into this CTA's shared memory
        for (int s = 0; s < C::kStages; ++s)
          if (issued & (1u << s)) wait_drain(B.full(s), (parities >> s) & 1u, ab, 2);
      }
    } else if (warp == 1) {
      // --------------------------------------------------------- MMA issuer
      // The whole warp follows the schedule, one elected lane issues a stage's MMAs
      // back to back; operand descriptors are built once for stage 0 and advanced
      // by the stage offset.
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
      for (int u = rs.first(); u >= 0; u = rs.next(u)) {
        const Unit t = unit(site(args, u), u);
        for (int kb = 0; kb < t.nkb; ++kb) {
          bool ok = wait(DV ? B.ready(r.idx) : B.full(r.idx), r.phase, ab, 3);
          ok = __all_sync(0xffffffffu, ok && wait(B.tempty(g.idx), g.phase ^ 1u, ab, 4));
          if (ok) {
            tc_fence_after();
            const uint32_t off = r.idx * C::kStageBytes;
            const uint32_t d = tmem + g.idx * C::kGroupCols;
            if (elect_one()) {   // one lane issues the stage's MMAs back to back
#pragma unroll
              for (int j = 0; j < C::kLeaves; ++j)   // fresh accumulator: one leaf
                mma_bf16(d + j * RP, desc_advance(adesc[j], off), desc_advance(wdesc[j], off), idesc, 0u);
              mma_commit(B.empty(r.idx));
              mma_commit(B.tfull(g.idx));
            }
            __syncwarp();
          }
          r.next<C::kStages>();
          g.next<C::kGroups>();
        }
      }
      if (elect_one()) mma_commit(B.drain());   // all MMAs issued above have completed ...
      __syncwarp();
      wait_drain(B.drain(), 0u, ab, 5);          // ... before TMEM is released or reused
    } else if (warp < 2 + C::kEpiWarps) {
      // ------------------------------------------------------------ epilogue
      const int q = warp & 3;                            // TMEM lane quarter this warp may access
      const int h = (warp - 2) >> 2;                     // column half
      const uint32_t tbase = tmem + (uint32_t(q * 32) << 16) + h * C::kCPT;
      Ring g;
      int k = 0;
      for (int u = rs.first(); u >= 0; u = rs.next(u), ++k) {
        const DownSite& S = site(args, u);
        const Unit t = unit(S, u);
        float stack[C::kLevels > 0 ? C::kLevels : 1][C::kCPT];
        float node[C::kCPT];
        bool ok_all = true;
#pragma unroll
        for (int i = 0; i < C::kGS; ++i) {
          if (i < t.nkb) {
            const bool ok = __all_sync(0xffffffffu, wait(B.tfull(g.idx), g.phase, ab, 6));   // warp-uniform: tcgen05.ld is .aligned
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
            if (ok && lane == 0) mbar_arrive(B.tempty(g.idx));
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
        const int row = t.mt * C::kBM + q * 32 + lane;
        if (ok_all && row < S.M) {
          float* __restrict__ part = S.part;
          float4* dst = reinterpret_cast<float4*>(part + (size_t(t.sl) * S.M + row) * RP + h * C::kCPT);
#pragma unroll
          for (int c = 0; c < C::kCPT; c += 4) dst[c / 4] = make_float4(node[c], node[c + 1], node[c + 2], node[c + 3]);
        }
        hook.stored(k);
      }
    } else if (warp < C::kWarps) {
      // ---------------------------------------------------- dV = bf16(dY*alpha)
      const int t = threadIdx.x - 32 * (2 + C::kEpiWarps);   // 0..127
      Ring r;
      for (int u = rs.first(); u >= 0; u = rs.next(u)) {
        const DownSite& S = site(args, u);
        const float alpha = S.alpha;
        const uint32_t a2 = pow2_bf16x2(alpha);
        const Unit tu = unit(S, u);
        for (int kb = 0; kb < tu.nkb; ++kb) {
          if (wait(B.full(r.idx), r.phase, ab, 7)) {
            if (!dv_is_dy(alpha)) {
              uint4* tile = reinterpret_cast<uint4*>(gbase + size_t(r.idx) * C::kStageBytes);
#pragma unroll
              for (int e = 0; e < C::kInBytes / 16 / 128; ++e) tile[t + 128 * e] = dv_bf16x8(tile[t + 128 * e], alpha, a2);
              fence_proxy_async();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(B.ready(r.idx));
          }
          r.next<C::kStages>();
        }
      }
    }
  }
};

// Fills in the unit bookkeeping of a launch's site table: n_mt, n_sl, u0, total.
template <int RP>
inline void down_units_of(DownArgs& args) {
  int u0 = 0;
  for (int i = 0; i < args.n; ++i) {
    DownSite& s = args.s[i];
    s.n_mt = int(ceil_div(s.M, 128));
    s.n_sl = int(ceil_div(s.Kred, down_slice(RP)));
    s.u0 = u0;
    u0 += s.n_mt * s.n_sl;
  }
  args.total = u0;
}

}  // namespace lora
