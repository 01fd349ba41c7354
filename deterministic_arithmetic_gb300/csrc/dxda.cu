// dxda.cu -- the two consumers of the finished dU rows in one launch (padded rank 16):
//   dX[m][k]   = fp32(sum_r du[m][r] * a[r][k])
//   dA partials: dA[r][k] = sum_m du[m][r] * x[m][k]   per 256-row chunk of M
// (page "[DSv4][P5-3] shared_grouped_lora_delta: CUDA + Triton, both
// batch-invariant", section "Summary": "dX = dU @ A, dA = dU^T @ X"; the combine
// launch that follows adds the chunk partials of dA with the canonical tree over
// chunks.)
//
// dX only writes (M x K FP32) and the dA partials only read (x, M x K BF16):
// as two launches each leaves one direction of the memory system idle. Here one
// pipeline does both per 128 x 128 tile of x: the producer streams the x tile,
// the a columns and the tile's 128 du rows into one shared-memory slot; the MMA
// issuer reads du twice, MN-major for the 8 dA leaves (x^T with du: M = 128
// columns, N = 16, K = 16 rows) and K-major for the dX expansion (du with a:
// M = 128 rows, N = 128 columns, K = 16), into one 256-column TMEM slot; the
// epilogue adds the dA leaves with the canonical tree and stores dX with TMA.
// Leaves, trees and rounding points are those of the separate up-projection
// (dX) and weight-gradient (dA) kernels: the outputs agree bit for bit.
//
// A unit is a 256-row chunk of M times a 128-column tile of K (two steps, one
// per 128-row half; one for a ragged last chunk of at most 128 rows). Units are
// dealt round robin to persistent CTAs, column tiles fastest, over all sites.
//
// Warp roles: 0 = TMA producer, 1 = MMA issuer (TMEM owner), 2..9 = epilogue
// (warp w: TMEM lanes 32 (w & 3) .. + 31, column half (w - 2) >> 2).
#include "common.cuh"
#include "kernels.h"

namespace lora {

namespace {

struct XaCfg {
  static constexpr int RP = 16;
  static constexpr int kBM = 128, kBK = 128;
  // slot: x [128 rows][128 columns] as two 64-row halves of two [64][64] boxes (128-byte swizzle),
  // a [RP][128] as two [RP][64] boxes (128-byte swizzle), du [128 rows][RP] (32-byte swizzle)
  static constexpr int kXBytes = kBM * kBK * 2;            // 32 KB
  static constexpr int kABytes = RP * kBK * 2;             // 4 KB
  static constexpr int kDuBytes = kBM * RP * 2;            // 4 KB
  static constexpr int kSlotBytes = kXBytes + kABytes + kDuBytes;   // 40 KB
  static constexpr int kSlots = 4;
  static constexpr int kLeaves = kBM / 16;                 // dA leaves per step
  static constexpr int kTCols = 256, kTSlots = 2;          // TMEM ring: 128 dA + 128 dX columns a slot
  static constexpr int kEpiWarps = 8;
  static constexpr int kThreads = 32 * (2 + kEpiWarps);
  static constexpr int kCPT = RP / 2;                      // dA columns of R per epilogue thread
  static constexpr int kStg = 1, kStgBytes = 32 * 32 * 4;  // dX staging boxes per epilogue warp (two measured slower)
  static constexpr size_t kStgOff = size_t(kSlots) * kSlotBytes;
  static constexpr size_t kArea = kStgOff + size_t(kEpiWarps) * kStg * kStgBytes;
  // mbarriers: slots (full, empty), TMEM (full, empty), drain, never
  static constexpr int kNumBars = 2 * kSlots + 2 * kTSlots + 2;
  static constexpr size_t kSmem = kArea + 1024 + kNumBars * 8 + 16;
  static_assert(kSlotBytes % 1024 == 0 && kStgOff % 1024 == 0, "1024-byte aligned tiles");
  static_assert(kWgradChunk == 2 * kBM, "a chunk is two steps");
  static_assert(kSmem <= 227 * 1024, "one CTA per SM");
};

// GR: a grouped launch (several sites); otherwise the table holds one site, read at fixed offsets
template <bool GR>
__global__ void __launch_bounds__(XaCfg::kThreads, 1)
    dxda_kernel(const __grid_constant__ Sites<XaSite, GR ? kMaxSites : 1> args, uint32_t* status) {
  using C = XaCfg;
  constexpr int RP = C::RP;
  auto site = [&](int u) -> const XaSite& {
    if constexpr (!GR) return args.s[0];
    int i = 0;
    while (i + 1 < args.n && u >= args.s[i + 1].u0) ++i;
    return args.s[i];
  };
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + C::kArea);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (C::kSlots + s); };
  auto tfull = [&](int t) { return bar0 + 8u * (2 * C::kSlots + t); };
  auto tempty = [&](int t) { return bar0 + 8u * (2 * C::kSlots + C::kTSlots + t); };
  const uint32_t drain = bar0 + 8u * (2 * C::kSlots + 2 * C::kTSlots), never = drain + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const uint32_t warp = warp_id(), lane = lane_id();
  const int total = args.total;
  // row tiles (halves) of a unit: 2, or 1 for a last chunk of at most 128 rows
  auto halves = [&](const XaSite& P, int ch) { return (min(P.M - ch * kWgradChunk, kWgradChunk) + C::kBM - 1) / C::kBM; };
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int t = 0; t < C::kTSlots; ++t) {
      mbar_init(tfull(t), 1);
      mbar_init(tempty(t), C::kEpiWarps);
    }
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0u;
    mbar_fence_init();
    for (int i = 0; i < args.n; ++i) {
      prefetch_map(&args.s[i].x);
      prefetch_map(&args.s[i].a);
      prefetch_map(&args.s[i].du);
      prefetch_map(&args.s[i].dx);
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
  const uint64_t pol_stream = policy_evict_first(), pol_keep = policy_evict_last();
  // the x tile [128 rows][128 columns] (two 64-row halves: columns 0..63, then 64..127) and the
  // a columns of one step into slot st
  auto copy_xa = [&](uint32_t st, uint32_t bar, const XaSite& P, int k0, int m0) {
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      tma_load(st + h2 * 16384u, &P.x, bar, k0, m0 + 64 * h2, pol_stream);
      tma_load(st + h2 * 16384u + 8192u, &P.x, bar, k0 + 64, m0 + 64 * h2, pol_stream);
    }
    tma_load(st + C::kXBytes, &P.a, bar, k0, 0, pol_keep);                 // a[0..RP)[k0 .. +63]
    tma_load(st + C::kXBytes + RP * 128, &P.a, bar, k0 + 64, 0, pol_keep); // a[0..RP)[k0+64 .. +127]
  };
  // x and a are inputs of the call and no output of the launches before this one, whose CTAs
  // start their dependents only after their own dependency wait, so every earlier writer of x
  // and a has completed when this kernel starts: the first ring slots get their x and a copies
  // before the dependency wait (while the predecessor's last CTAs finish), their du rows (the
  // predecessor's output) after it. Not with a test hook set: the stall comes first.
  int pre = 0;
  if (warp == 0 && lane == 0 && !stall_requested(status, kKindWgrad) && !stall_requested(status, kKindUp)) {
    for (int u = blockIdx.x; u < total && pre < C::kSlots; u += gridDim.x) {
      const XaSite& P = site(u);
      const int kt = (u - P.u0) % P.n_kt, ch = (u - P.u0) / P.n_kt;
      for (int hh = 0; hh < halves(P, ch) && pre < C::kSlots; ++hh, ++pre) {
        mbar_expect_tx(full(pre), uint32_t(C::kSlotBytes));   // fresh slots: free, phase 0
        copy_xa(base + pre * C::kSlotBytes, full(pre), P, kt * C::kBK, ch * kWgradChunk + hh * C::kBM);
      }
    }
  }
  grid_dependency_wait();      // predecessor done: the du rows are complete
  grid_dependents_launch();
  const Abort ab = make_abort(abort_flag, status);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      if (stall_requested(status, kKindWgrad)) stall_wait(never, ab, 29);   // test hooks: a wait that runs out
      if (stall_requested(status, kKindUp)) stall_wait(never, ab, 10);
      Ring r;
      uint32_t issued = 0, parities = 0;
      int i = 0;   // step index of this CTA
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const XaSite& P = site(u);
        const int kt = (u - P.u0) % P.n_kt, ch = (u - P.u0) / P.n_kt;
        const int k0 = kt * C::kBK;
        for (int hh = 0; hh < halves(P, ch); ++hh, ++i) {
          const int s = int(r.idx);
          const uint32_t st = base + s * C::kSlotBytes;
          const int m0 = ch * kWgradChunk + hh * C::kBM;
          if (i < pre) {   // slot i, phase 0: its x and a copies are in flight
            issued |= 1u << s;
            tma_load(st + C::kXBytes + C::kABytes, &P.du, full(s), 0, m0, pol_keep);   // du rows m0 .. +127
          } else if (wait(empty(s), r.phase ^ 1u, ab, 81)) {
            mbar_expect_tx(full(s), uint32_t(C::kSlotBytes));
            issued |= 1u << s;
            parities = (parities & ~(1u << s)) | (r.phase << s);
            copy_xa(st, full(s), P, k0, m0);
            tma_load(st + C::kXBytes + C::kABytes, &P.du, full(s), 0, m0, pol_keep);   // du rows m0 .. +127
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
    constexpr uint32_t idesc_da = idesc_bf16(128, RP, 1, 1);    // x^T MN-major, du MN-major
    constexpr uint32_t idesc_dx = idesc_bf16(128, 128, 0, 1);   // du K-major, a MN-major
    const uint32_t du0 = base + uint32_t(C::kXBytes + C::kABytes);
    uint64_t a_da[C::kLeaves], b_da[C::kLeaves];
#pragma unroll
    for (int j = 0; j < C::kLeaves; ++j) {
      // dA leaf j: x rows 16j..16j+15 (64-row half j/4), transposed view: MN-major, 128-byte swizzle,
      // 64-column blocks 8 KB apart, 8-row groups 1 KB apart
      a_da[j] = smem_desc(base + (j >> 2) * 16384u + (j & 3) * 2048u, 8192u, 1024u, kLayoutSW128);
      // du rows 16j..16j+15 of [128 m][16 r]: MN-major (r contiguous), 32-byte swizzle
      b_da[j] = smem_desc(du0 + j * 512u, 256u, 256u, kLayoutSW32);
    }
    const uint64_t a_dx = smem_desc(du0, 16u, 256u, kLayoutSW32);                              // du K-major
    const uint64_t b_dx = smem_desc(base + uint32_t(C::kXBytes), RP * 128u, 1024u, kLayoutSW128);   // a MN-major
    Ring r, t;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const XaSite& P = site(u);
      const int ch = (u - P.u0) / P.n_kt;
      for (int hh = 0; hh < halves(P, ch); ++hh) {
        bool ok = wait(full(r.idx), r.phase, ab, 83);
        ok = __all_sync(0xffffffffu, ok && wait(tempty(t.idx), t.phase ^ 1u, ab, 84));
        if (ok) {
          tc_fence_after();
          const uint32_t off = r.idx * C::kSlotBytes;
          const uint32_t d = tmem + t.idx * C::kTCols;
          if (elect_one()) {   // one lane issues the step's MMAs back to back
#pragma unroll
            for (int j = 0; j < C::kLeaves; ++j)
              mma_bf16(d + j * RP, desc_advance(a_da[j], off), desc_advance(b_da[j], off), idesc_da, 0u);
            mma_bf16(d + 128u, desc_advance(a_dx, off), desc_advance(b_dx, off), idesc_dx, 0u);
            mma_commit(empty(r.idx));
            mma_commit(tfull(t.idx));
          }
          __syncwarp();
        }
        r.next<C::kSlots>();
        t.next<C::kTSlots>();
      }
    }
    if (elect_one()) mma_commit(drain);
    __syncwarp();
    wait_drain(drain, 0u, ab, 86);
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;                        // column half of R (dA); of the tile (dX)
    const uint32_t tq = tmem + (uint32_t(q * 32) << 16);
    const int tr = q * 32 + lane;                         // TMEM lane: row (dX) or column (dA)
    const uint32_t stg0 = base + uint32_t(C::kStgOff) + (warp - 2) * C::kStg * C::kStgBytes;
    uint8_t* stg_ptr = gbase + C::kStgOff + (warp - 2) * C::kStg * C::kStgBytes;
    const uint64_t pol_out = policy_evict_first();
    Ring t;
    int sidx = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const XaSite& P = site(u);
      const int kt = (u - P.u0) % P.n_kt, ch = (u - P.u0) / P.n_kt;
      const int nh = halves(P, ch), K = P.K;
      float da_first[C::kCPT];
      bool ok_all = true;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float dan[C::kCPT];
        if (hh < nh) {
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
          const int row0 = ch * kWgradChunk + hh * C::kBM + q * 32;
#pragma unroll
          for (int bx = 0; bx < 2; ++bx) {
            const int col0 = h * 64 + bx * 32;
            const int gcol = kt * C::kBK + col0;
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
              if (ok && row0 < P.M) tma_store(&P.dx, stg0 + sidx * C::kStgBytes, gcol, row0, pol_out);
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
          const int col = kt * C::kBK + tr;
          if (ok_all && col < K) {
            float* dst = P.da_part + (size_t(ch) * RP + h * C::kCPT) * K + col;
#pragma unroll
            for (int c = 0; c < C::kCPT; ++c) dst[size_t(c) * K] = __fadd_rn(da_first[c], dan[c]);
          }
        }
      }
    }
    if (lane == 0) tma_store_wait_all<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_dxda(XaArgs& args, uint32_t* status, int grid, cudaStream_t st) {
  using C = XaCfg;
  if (args.n < 1 || args.n > kMaxSites) return cudaErrorInvalidValue;
  int u0 = 0;
  for (int i = 0; i < args.n; ++i) {
    XaSite& s = args.s[i];
    s.n_kt = int(ceil_div(s.K, C::kBK));
    s.n_ch = int(ceil_div(s.M, kWgradChunk));
    s.u0 = u0;
    u0 += s.n_kt * s.n_ch;
  }
  args.total = u0;
  if (args.n > 1) return launch_pdl(dxda_kernel<true>, dim3(grid), dim3(C::kThreads), C::kSmem, st, args, status);
  return launch_pdl(dxda_kernel<false>, dim3(grid), dim3(C::kThreads), C::kSmem, st, first_site(args), status);
}

cudaError_t prepare_dxda() {
  const cudaError_t e = cudaFuncSetAttribute(dxda_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(XaCfg::kSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(dxda_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(XaCfg::kSmem));
}

}  // namespace lora
