// up_phase.cuh -- the rank-R expansions (write-bound), as a kernel phase:
//   forward : dY_lora[m][n] = fp32(sum_r u[m][r] * b[n][r]) * alpha    ("(U @ B^T) * alpha")
//   backward: dX[m][k] = fp32(sum_r du[m][r] * a[r][k])                ("dX = dU @ A")
// (page "[DSv4][P5-3] shared_grouped_lora_delta: CUDA + Triton, both
// batch-invariant", section "Summary"; the alpha scale is fused into the
// epilogue, as that page's "Benchmark" section proposes.)
//
// The producer loads a unit's finished u / du rows (TMA) once the `rows`
// policy says they are there: at once in a standalone launch (the rows kernel
// before it wrote them), after the row tile's ready flag in the fused forward.
// Work unit = (128-row tile, BN-column tile), BN = 256 / (RP / 16), units dealt
// out round robin, so that at any time the CTAs write one compact band of the
// output (consecutive units are neighbours in memory), which the memory
// system absorbs markedly faster than each CTA writing its own distant region.
// The unit is one tcgen05 MMA per 16-wide slice of R (M=128, N=BN, K=16), each
// into its own TMEM accumulator, summed by the canonical tree. Eight epilogue
// warps read TMEM, finish the tree (and the alpha multiply); each warp stages
// its own 32 x 32 FP32 boxes in 128-byte-swizzled shared memory (a ring of
// four, no barrier across warps) and writes them with TMA stores (L2
// evict-first), so every output byte is written exactly once, in full lines.
//
// YBF (forward only): dY_lora is written as BF16, bf16(fp32(sum) * alpha): the
// FP32 value rounded once more (round to nearest even), half the bytes. Each
// 32-column box is then 32 rows x 64 bytes (64-byte swizzle).
//
// Warp roles: 0 = TMA producer (u / du rows, B / A weight tile), 1 = MMA
// issuer (TMEM owner), 2..9 = epilogue.
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "sched.cuh"

namespace lora {

template <int RP, bool DX>
struct UpCfg {
  static constexpr int kBM = 128;
  static constexpr int kLeaves = RP / 16;
  static constexpr int kBN = up_bn(RP);
  static constexpr int kSpan = RP * 2;                 // bytes of one operand row (r contiguous)
  static constexpr int kABytes = kBM * RP * 2;         // U / dU tile [128][RP]
  static constexpr int kBBytes = kBN * RP * 2;         // B tile [BN][RP] or A tile [RP][BN]
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = RP == 16 ? 6 : (RP == 32 ? 5 : 3);   // operand ring (weight tile from L2)
  static constexpr int kBufCols = kLeaves * kBN;       // 256 TMEM columns per buffer
  static constexpr int kBufs = 512 / kBufCols;
  static constexpr int kEpiWarps = 8;
  static constexpr int kWarps = 2 + kEpiWarps;
  static constexpr int kHalfCols = kBN / 2;
  static constexpr int kChunk = 32;                    // FP32 columns per TMA store box (128 bytes)
  static constexpr int kChunks = kHalfCols / kChunk;
  static constexpr int kCols = kLeaves == 1 ? 64 : (kLeaves == 2 ? 32 : 16);   // TMEM columns per load round
  static constexpr int kBoxes = kCols >= kChunk ? kCols / kChunk : 1;           // store boxes per round group
  static constexpr int kRounds = kCols >= kChunk ? 1 : kChunk / kCols;          // load rounds per box group
  static constexpr int kStg = 4;                       // staging buffers per epilogue warp
  static constexpr int kStgBytes = 32 * kChunk * 4;    // one 32-row x 32-column FP32 box: 4 KB
  static constexpr size_t kStgOff = size_t(kStages) * kStageBytes;
  static constexpr size_t kBarOff = kStgOff + size_t(kEpiWarps) * kStg * kStgBytes;
  static constexpr size_t kArea = kBarOff;             // stage ring + staging, from the 1024-byte aligned base
  static constexpr int kNumBars = 2 * kStages + 2 * kBufs + 2;   // ring, TMEM ring, drain, never
  static_assert(kStageBytes % 1024 == 0, "tiles must stay 1024-byte aligned");
  static_assert(kBufs == 2, "double-buffered accumulators");
};

// Rows policy of a standalone launch: the rows are complete when it starts.
struct RowsDone {
  __device__ __forceinline__ bool ready(const UpSite&, int, const Abort&) const { return true; }
};

template <int RP, bool DX, bool YBF, bool GR>
struct UpPhase {
  using C = UpCfg<RP, DX>;
  using Args = Sites<UpSite, GR ? kMaxSites : 1>;
  static_assert(!(DX && YBF), "BF16 output is the forward's");

  struct Bars {
    uint32_t b0;
    __device__ __forceinline__ uint32_t full(int s) const { return b0 + 8u * s; }              // rows + weight tile landed
    __device__ __forceinline__ uint32_t empty(int s) const { return b0 + 8u * (C::kStages + s); }  // stage free (MMA done)
    __device__ __forceinline__ uint32_t tfull(int b) const { return b0 + 8u * (2 * C::kStages + b); }
    __device__ __forceinline__ uint32_t tempty(int b) const { return b0 + 8u * (2 * C::kStages + C::kBufs + b); }
    __device__ __forceinline__ uint32_t drain() const { return b0 + 8u * (2 * C::kStages + 2 * C::kBufs); }
    __device__ __forceinline__ uint32_t never() const { return drain() + 8u; }   // completed by nothing
  };

  // site of unit u (sites are few and ordered by first unit)
  static __device__ __forceinline__ const UpSite& site(const Args& args, int u) {
    if constexpr (!GR) return args.s[0];
    int i = 0;
    while (i + 1 < args.n && u >= args.s[i + 1].u0) ++i;
    return args.s[i];
  }

  // thread 0, before the kernel's mbarrier init fence
  static __device__ void init(const Bars& B, const Args& args) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(B.full(s), 1);
      mbar_init(B.empty(s), 1);
    }
    for (int b = 0; b < C::kBufs; ++b) {
      mbar_init(B.tfull(b), 1);
      mbar_init(B.tempty(b), C::kEpiWarps);
    }
    mbar_init(B.drain(), 1);
    mbar_init(B.never(), 1);
    for (int i = 0; i < (GR ? args.n : 1); ++i) {
      prefetch_map(&args.s[i].a);
      prefetch_map(&args.s[i].b);
      prefetch_map(&args.s[i].out);
    }
  }

  // All warps of the phase call this (warps beyond kWarps return at once). `base`: 1024-byte
  // aligned start of the phase's shared memory (generic pointer gbase). Returns when every copy,
  // MMA and store the phase issued has completed.
  template <class Rows>
  static __device__ void run(const Args& args, uint8_t* gbase, uint32_t base, const Bars& B, uint32_t tmem,
                             const Abort& ab, const uint32_t* status, const StaticSched sched, const Rows& rows) {
    const uint32_t warp = warp_id(), lane = lane_id();
    const uint32_t stg0 = base + uint32_t(C::kStgOff);               // staging buffers [epilogue warp][kStg]
    uint8_t* stg_ptr = gbase + C::kStgOff;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      if (stall_requested(status, kKindUp)) stall_wait(B.never(), ab, 10);   // test hook: a wait that runs out
      const uint64_t pol = policy_evict_last();
      Ring r;
      uint32_t issued = 0, parities = 0;
      for (int u = sched.first(); u >= 0; u = sched.next(u)) {
        const UpSite& P = site(args, u);
        const int mt = (u - P.u0) / P.n_nt, nt = (u - P.u0) % P.n_nt;
        if (wait(B.empty(r.idx), r.phase ^ 1u, ab, 11) && rows.ready(P, mt, ab)) {
          const uint32_t st = base + r.idx * C::kStageBytes;
          mbar_expect_tx(B.full(r.idx), C::kStageBytes);
          tma_load(st, &P.a, B.full(r.idx), 0, mt * C::kBM, pol);                     // u / du rows of the tile
          if (DX) {
#pragma unroll
            for (int i = 0; i < C::kBN / 64; ++i)                                  // a[0..RP)[k..k+63]
              tma_load(st + C::kABytes + i * (RP * 128), &P.b, B.full(r.idx), nt * C::kBN + 64 * i, 0, pol);
          } else {
            tma_load(st + C::kABytes, &P.b, B.full(r.idx), 0, nt * C::kBN, pol);     // b rows n..n+BN
          }
          issued |= 1u << r.idx;
          parities = (parities & ~(1u << r.idx)) | (r.phase << r.idx);
        }
        r.next<C::kStages>();
      }
      for (int s = 0; s < C::kStages; ++s)
        if (issued & (1u << s)) wait_drain(B.full(s), (parities >> s) & 1u, ab, 12);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, C::kBN, 0, DX ? 1 : 0);
      constexpr uint32_t lay = layout_for_span(C::kSpan);
      Ring r, b;
      for (int u = sched.first(); u >= 0; u = sched.next(u)) {
        bool ok = wait(B.full(r.idx), r.phase, ab, 13);
        ok = ok && wait(B.tempty(b.idx), b.phase ^ 1u, ab, 14);
        if (ok) {
          tc_fence_after();
          const uint32_t st = base + r.idx * C::kStageBytes;
#pragma unroll
          for (int j = 0; j < C::kLeaves; ++j) {
            // u/du tile: K-major, rows of RP*2 bytes, swizzle span = row; K step j = +32 bytes
            const uint64_t adesc = smem_desc(st + 32u * j, 16u, 8u * C::kSpan, lay);
            uint64_t bdesc;
            if (DX)   // a tile: 64-column blocks [RP rows][64 k], MN-major, 128-byte swizzle; K step = 16 rows
              bdesc = smem_desc(st + C::kABytes + j * 2048u, RP * 128u, 1024u, kLayoutSW128);
            else      // b tile [BN rows][RP]: K-major like the u tile
              bdesc = smem_desc(st + C::kABytes + 32u * j, 16u, 8u * C::kSpan, lay);
            mma_bf16(tmem + b.idx * C::kBufCols + j * C::kBN, adesc, bdesc, idesc, 0u);
          }
          mma_commit(B.empty(r.idx));
          mma_commit(B.tfull(b.idx));
        }
        r.next<C::kStages>();
        b.next<C::kBufs>();
      }
      mma_commit(B.drain());                 // every MMA issued above has completed ...
      wait_drain(B.drain(), 0u, ab, 17);     // ... before TMEM is released
    }
  } else if (warp < 2 + C::kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const uint32_t trow = tmem + (uint32_t(q * 32) << 16);
    const uint32_t my_stg = stg0 + (warp - 2) * C::kStg * C::kStgBytes;
    const uint64_t pol_out = policy_evict_first();
    uint8_t* my_stg_ptr = stg_ptr + (warp - 2) * C::kStg * C::kStgBytes;
    int sidx = 0;
    Ring b;
    for (int u = sched.first(); u >= 0; u = sched.next(u)) {
      const UpSite& P = site(args, u);
      const int mt = (u - P.u0) / P.n_nt, nt = (u - P.u0) % P.n_nt;
      const int M = P.M, Nout = P.Nout;
      const float alpha = P.alpha;
      const bool ok = __all_sync(0xffffffffu, wait(B.tfull(b.idx), b.phase, ab, 15));
      tc_fence_after();
      // one TMEM round trip per group of kBoxes 32-column boxes (64 registers of leaves per round)
#pragma unroll
      for (int grp = 0; grp < C::kChunks / C::kBoxes; ++grp) {
        const int col0 = h * C::kHalfCols + grp * C::kBoxes * C::kChunk;
        if (nt * C::kBN + col0 >= Nout) break;                       // uniform over the column half
        if (lane == 0) tma_store_wait_read<C::kStg - C::kBoxes>();   // these buffers' previous stores have read them
        __syncwarp();
#pragma unroll
        for (int rd = 0; rd < C::kRounds; ++rd) {
          uint32_t v[C::kLeaves][C::kCols / 8][8];
#pragma unroll
          for (int j = 0; j < C::kLeaves; ++j)
#pragma unroll
            for (int b8 = 0; b8 < C::kCols / 8; ++b8)
#pragma unroll
              for (int e = 0; e < 8; ++e) v[j][b8][e] = 0u;
          if (ok) {
#pragma unroll
            for (int j = 0; j < C::kLeaves; ++j)
#pragma unroll
              for (int b8 = 0; b8 < C::kCols / 8; ++b8)
                tmem_ld8(trow + b.idx * C::kBufCols + j * C::kBN + col0 + rd * C::kCols + b8 * 8, v[j][b8]);
            tmem_ld_wait();
          }
#pragma unroll
          for (int j = 0; j < C::kLeaves; ++j)
#pragma unroll
            for (int b8 = 0; b8 < C::kCols / 8; ++b8) reg_fence(v[j][b8]);
          // leaf tree of column e of this round (and the alpha multiply of the forward)
          auto value = [&](int e) {
            const int b8 = e / 8, k = e % 8;
            float s;
            if (C::kLeaves == 1) s = __uint_as_float(v[0][b8][k]);
            else if (C::kLeaves == 2) s = __fadd_rn(__uint_as_float(v[0][b8][k]), __uint_as_float(v[1][b8][k]));
            else s = tree4(__uint_as_float(v[0][b8][k]), __uint_as_float(v[1][b8][k]), __uint_as_float(v[2][b8][k]),
                           __uint_as_float(v[3][b8][k]));
            return DX ? s : __fmul_rn(s, alpha);
          };
          if constexpr (YBF) {
#pragma unroll
            for (int e8 = 0; e8 < C::kCols / 8; ++e8) {
              const int gcol = rd * C::kCols + e8 * 8;                // column within the group
              const int box = gcol / C::kChunk, cc = (gcol % C::kChunk) / 8;
              float f[8];
#pragma unroll
              for (int t8 = 0; t8 < 8; ++t8) f[t8] = value(e8 * 8 + t8);
              // 32 rows x 32 BF16 columns per box: 64-byte rows, 64-byte swizzle, chunk ^ ((row / 2) % 4)
              uint8_t* buf = my_stg_ptr + ((sidx + box) % C::kStg) * C::kStgBytes + lane * 64;
              *reinterpret_cast<uint4*>(buf + ((cc ^ ((lane >> 1) & 3)) * 16)) = pack_bf16x8(f);
            }
          } else {
#pragma unroll
            for (int e4 = 0; e4 < C::kCols / 4; ++e4) {
              const int gcol = rd * C::kCols + e4 * 4;                // column within the group
              const int box = gcol / C::kChunk, cc = (gcol % C::kChunk) / 4;
              // each warp stages its own 32 rows x 32 columns: 128-byte swizzle, chunk ^ (row % 8)
              uint8_t* buf = my_stg_ptr + ((sidx + box) % C::kStg) * C::kStgBytes + lane * 128;
              *reinterpret_cast<float4*>(buf + ((cc ^ (lane & 7)) * 16)) =
                  make_float4(value(e4 * 4), value(e4 * 4 + 1), value(e4 * 4 + 2), value(e4 * 4 + 3));
            }
          }
        }
        fence_proxy_async();
        __syncwarp();
        const int row0 = mt * C::kBM + q * 32;
        if (lane == 0) {
          // one bulk group per staging buffer, empty when the box lies past M or N, so that
          // "at most kStg - kBoxes groups pending" always frees exactly the buffers reused next
#pragma unroll
          for (int box = 0; box < C::kBoxes; ++box) {
            const int ncol = nt * C::kBN + col0 + box * C::kChunk;
            if (ok && row0 < M && ncol < Nout)
              tma_store(&P.out, my_stg + ((sidx + box) % C::kStg) * C::kStgBytes, ncol, row0, pol_out);
            tma_store_commit();
          }
        }
        sidx = (sidx + C::kBoxes) % C::kStg;
      }
      tc_fence_before();
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(B.tempty(b.idx));
      b.next<C::kBufs>();
    }
    if (lane == 0) tma_store_wait_all<0>();
  }

  }
};

// Fills in the unit bookkeeping of a launch's site table: n_mt, n_nt, u0, total.
template <int RP>
inline void up_units_of(UpArgs& args) {
  int u0 = 0;
  for (int i = 0; i < args.n; ++i) {
    UpSite& s = args.s[i];
    s.n_mt = int(ceil_div(s.M, 128));
    s.n_nt = int(ceil_div(s.Nout, up_bn(RP)));
    s.u0 = u0;
    u0 += s.n_mt * s.n_nt;
  }
  args.total = u0;
}

}  // namespace lora
