// kernels.h -- internal interface between the C ABI (api.cu) and the kernel
// translation units. Not installed; the public interface is include/lora_delta.h.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lora {

// Rank R is padded to RP in {16, 32, 64} inside the kernels (tcgen05 needs N
// and K to be multiples of 16); padded rows/columns are TMA zero fill.
constexpr int padded_rank(int R) { return R <= 16 ? 16 : (R <= 32 ? 32 : 64); }

// Down-projection (U, dU): the reduction over K (or N) is cut into slices of
// this many elements; each slice is one work unit and leaves one FP32 partial.
// Slices hold a power-of-two number of 16-element leaves, so the canonical
// tree over all leaves does not depend on the slice length.
constexpr int down_slice(int RP) { return RP == 64 ? 256 : 1024; }
// Weight gradients (dA, dB): rows of the batch are cut into fixed chunks.
constexpr int kWgradChunk = 256;
// Fused dU + dB pass over dY (R <= 16): 512-column slices of N (dU partials)
// and 256-row chunks of M (dB partials).
constexpr int kDySlice = 512, kDyChunk = 256;
// Slices the dU partials of the backward pass are cut into (ranks <= 16 use the fused pass).
constexpr int du_slice(int RP) { return RP == 16 ? kDySlice : down_slice(RP); }
// Up-projection tile width (N direction) per padded rank.
constexpr int up_bn(int RP) { return 256 / (RP / 16); }

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Grouped launches: every kernel takes a table of up to kMaxSites independent
// problems ("sites", e.g. the fc1 and fc2 LoRA insertion points of one MLP),
// all of the same padded rank, and deals their work units out as one unit
// space: site i owns units [u0, u0 + its unit count). A single-site call is a
// table of one. The table is a __grid_constant__ kernel parameter, so its
// tensor maps stay in parameter space (what TMA needs) when indexed by site.
constexpr int kMaxSites = 4;
// A table of NS sites (NS = kMaxSites for grouped launches, 1 otherwise: a
// smaller parameter block per launch). R: the rank (up-projection only).
template <class Site, int NS>
struct Sites {
  Site s[NS];
  int n, total, R;
};
// The one-site table of a launch built as a kMaxSites table.
template <class Site>
inline Sites<Site, 1> first_site(const Sites<Site, kMaxSites>& a) {
  Sites<Site, 1> b;
  b.s[0] = a.s[0];
  b.n = 1;
  b.total = a.total;
  b.R = a.R;
  return b;
}

// Down-projection (U or, with dV, dU partials): reduction over Kred in slices.
struct DownSite {
  CUtensorMap in, w;   // input rows (X or dY, boxes 128 x 32) and weight (A [R][Kred] or B [Kred][R])
  float* part;         // [n_sl][M][RP] slice partials
  int M, Kred, n_mt, n_sl, u0;
  float alpha;         // dV = bf16(dY * alpha) (dV launches)
};
using DownArgs = Sites<DownSite, kMaxSites>;

// Up-projection (dY_lora, or dX) from the finished u / du rows.
struct UpSite {
  CUtensorMap a, b, out;   // u / du rows (box 128 x RP), weight (B rows or A columns), output
  int M, Nout, n_mt, n_nt, u0;
  float alpha;             // forward scale (1 for dX)
};
using UpArgs = Sites<UpSite, kMaxSites>;

// Fused dU + dB pass over dY (R <= 16).
struct DySite {
  CUtensorMap dy, b, u;   // dY rows (boxes 128 x 32), b rows, u rows (boxes 128 x RP)
  float* du_part;         // [n_sl][M][RP]
  float* db_part;         // [n_ch][RP][N]
  int M, N, n_sl, n_ch, u0;
  float alpha;
};
using DyArgs = Sites<DySite, kMaxSites>;

// Weight-gradient chunk partials (dA from X and du; dB from dY and u for R > 16).
struct WgSite {
  CUtensorMap in, g;      // wide operand (X or dY, boxes 64 x 64) and du / u rows (boxes 64 x RP)
  float* part;            // [n_ch][RP][Cw]
  int M, Cw, n_ct, n_ch, u0;
  float alpha;            // dV = bf16(dY * alpha) (dB launches)
};
using WgArgs = Sites<WgSite, kMaxSites>;

// dX and the dA chunk partials from the finished du rows in one pass (padded rank 16).
struct XaSite {
  CUtensorMap x, a, du, dx;   // x 64 x 64 and a RP x 64 boxes (128-byte swizzle); du 128 x RP (row span);
                              // dx 32 x 32 FP32 (128-byte swizzle)
  float* da_part;             // [n_ch][RP][K]
  int M, K, n_kt, n_ch, u0;
};
using XaArgs = Sites<XaSite, kMaxSites>;

// Launch with programmatic stream serialization (the kernel calls
// grid_dependency_wait() before its first global-memory access).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Work-unit counts (all launches use persistent CTAs over units).
inline int64_t down_units(int64_t M, int64_t Kred, int RP) { return ceil_div(M, 128) * ceil_div(Kred, down_slice(RP)); }
inline int64_t up_units(int64_t M, int64_t Nout, int RP) { return ceil_div(M, 128) * ceil_div(Nout, up_bn(RP)); }
inline int64_t wgrad_units(int64_t M, int64_t C, int RP) { (void)RP; return ceil_div(M, kWgradChunk) * ceil_div(C, 128); }

// Launchers (return the launch error, if any). `status` is the device status
// word; `grid` the number of persistent CTAs.
// args: sites filled in except n_mt, n_sl, u0 and total (set here)
cudaError_t launch_down(int RP, bool dv, DownArgs& args, uint32_t* status, int grid, cudaStream_t st);
// up: a = u / du rows (box 128 x RP), complete when the launch starts (written by the preceding
// rows kernel); y_bf16 (forward only): `out` is a BF16 dY_lora map with 32 x 32 boxes, 64-byte
// swizzle. args: sites filled in except n_mt, n_nt, u0 and total (set here).
cudaError_t launch_up(int RP, bool dx, bool y_bf16, UpArgs& args, uint32_t* status, int grid, cudaStream_t st);
// args: sites filled in except n_sl, n_ch, u0 and total (set here)
cudaError_t launch_dy(DyArgs& args, uint32_t* status, int grid, cudaStream_t st);
// args: sites filled in except n_ct, n_ch, u0 and total (set here)
cudaError_t launch_wgrad(int RP, bool dv, WgArgs& args, uint32_t* status, int grid, cudaStream_t st);

// du: complete when the launch starts (written by the preceding kernel). args: sites filled in
// except n_kt, n_ch, u0 and total (set here).
cudaError_t launch_dxda(XaArgs& args, uint32_t* status, int grid, cudaStream_t st);
inline int64_t dxda_units(int64_t M, int64_t K) { return ceil_div(M, kWgradChunk) * ceil_div(K, 128); }

// The BF16 rows of U (or dU) from the slice partials of the down (or dy) kernel: for every row
// and every group of 8 columns, the canonical pairwise tree over the S slice partials, rounded
// to BF16. One thread per group of 8 values, all sites of a call in one launch.
struct RowsSite {
  const float* part;       // [S][M][RP]
  __nv_bfloat16* out;      // [M][R]
  int M, S;
  int64_t item0;           // first item of this site (M * R / 8 items per site)
};
struct RowsArgs {
  RowsSite s[kMaxSites];
  int64_t total;
  int n, R, RP;
};


// Single-launch forward of one site (fwd_fused.cu): the down, rows and up steps, ordered by
// claimed work. ctl: the control words (kFusedCtlWords, zero between launches); batches of up to
// kFusedMaxTiles row tiles of 128 rows.
constexpr int kFusedMaxTiles = 4096;
constexpr int kFusedCtlWords = 4 + 2 * kFusedMaxTiles;
cudaError_t launch_fwd_fused(int RP, bool y_bf16, DownArgs& dargs, UpArgs& uargs, __nv_bfloat16* u, int R,
                             uint32_t* ctl, int nsm, uint32_t* status, cudaStream_t st);
cudaError_t prepare_fwd_fused();

// Single-launch forward of one site on thread-block clusters (fwd_cluster.cu), padded ranks 16 and
// 32: a cluster of cl CTAs owns a 128-row tile at a time, each CTA a share of its K-slices and of
// its column tiles; the slice partials meet through the workspace, ordered by mbarriers at cluster
// scope. Column tiles of the expansion are fc_bn(RP) wide.
constexpr int fc_bn(int RP) { return 128 / (RP / 16); }
struct FcArgs {
  CUtensorMap x, a, b, out;   // x boxes 128 x 32 (64-byte swizzle); a RP x 64 (128-byte); b fc_bn x RP (row span); out 32 x 32
  float* part;                // [S][M][RP] slice partials
  __nv_bfloat16* u;           // [M][R]
  int M, K, N, R, S, n_mt, n_nt;   // S, n_mt, n_nt: set by the launcher
  float alpha;
};
// up = false: the down-projection and the U rows only (the up-projection launch follows; y_bf16 and
// the b and out maps are then unused).
cudaError_t launch_fwd_cluster(int RP, bool y_bf16, bool up, FcArgs& a, uint32_t* status, int cl, int ncl,
                               cudaStream_t st);
// Clusters of cl CTAs of that instance that fit on the device at once.
cudaError_t fwd_cluster_max_clusters(int RP, bool y_bf16, bool up, int cl, int* n);
cudaError_t prepare_fwd_cluster();

// Backward of one site (padded rank 16) on thread-block clusters (bwd_cluster.cu): a cluster of cl
// CTAs owns a 256-row chunk at a time; each CTA a share of its 512-column dU slices (phase A: dU
// and dB partials from one pass over dY), then, after the cluster has met and every CTA holds the
// chunk's dU rows, a share of its 128-column tiles of K (phase C: dX and the dA chunk partials).
struct BcArgs {
  CUtensorMap dy, b, u, x, a, dx;   // dy 128 x 32 (64-byte swizzle); b, u 128 x RP (row span); x 64 x 64 and
                                    // a RP x 64 (128-byte); dx 32 x 32 FP32 (128-byte)
  float* du_part;                   // [S][M][RP] dU slice partials
  float* db_part;                   // [C][RP][N] dB chunk partials
  float* da_part;                   // [C][RP][K] dA chunk partials
  __nv_bfloat16* du;                // [M][R]
  int M, K, N, R, S, n_ch, n_kt;    // S, n_ch, n_kt: set by the launcher
  float alpha;
  // Rows per unit (phase_c false only; 256 with phase C): 256, a chunk, or 128, one row tile, whose
  // dB tree is then the unit's partial -- db_part holds ceil(M / unit_rows) partials, and the
  // combine's canonical tree over them first adds the two tiles of each chunk.
  int unit_rows;
};
// phase_c = false: phase A and the dU rows only (the dX, dA and combine launches follow; the x, a
// and dx maps are then unused).
cudaError_t launch_bwd_cluster(bool phase_c, BcArgs& a, uint32_t* status, int cl, int ncl, cudaStream_t st);
cudaError_t bwd_cluster_max_clusters(bool phase_c, int cl, int* n);
cudaError_t prepare_bwd_cluster();

// Final combine of the weight-gradient chunk partials: canonical tree over
// the C chunks, FP32 out. part is [C][RP][cols] (cols = K for dA, N for dB).
struct CombineJob {
  const float* part;
  float* out;
  int C;               // number of chunk partials
  int cols;            // K (dA) or N (dB); a multiple of 8
  int R, RP;           // rank and padded rank
  int transpose;       // 0: out[R][cols] (dA); 1: out[cols][R] (dB)
};
struct CombineJobs {
  CombineJob j[2 * kMaxSites];   // dA and dB of every site
  int n;
};
cudaError_t launch_combine(const CombineJobs& jobs, cudaStream_t st);
// The rows launch (rows.cu); jobs (may be null): combine jobs run by the same launch after the
// rows blocks (the backward's dB, whose chunk partials the preceding kernel has just written).
cudaError_t launch_rows(RowsArgs& args, const CombineJobs* jobs, int nsm, cudaStream_t st);

// dV = bf16(fp32(dy * alpha)) from a binary32 dY of n values (n a multiple of 8), into dv.
cudaError_t launch_dv_from_f32(const float* dy, float alpha, int64_t n, void* dv, int nsm, cudaStream_t st);

// Exact mode of the weight gradients (exact.cu): per output, kDigits signed 64-bit digits in radix
// 2^32 (digit i weighs 2^(32 i - 266)) and three counters (+inf, -inf, NaN products): kExactSlots.
constexpr int kDigits = 18, kExactSlots = kDigits + 3;
// The digit kernel runs at most kMaxExactGrid persistent CTAs; exact_part_bytes is its scratch
// (segment records and digit arrays) for a P x Q output.
constexpr int kMaxExactGrid = 512;
size_t exact_part_bytes(int64_t M, int64_t P, int64_t Q);
// sum_m left[m][p] * right[m][q] (right = bf16(fp32(dy * alpha)) with dv) for p < P, q < Q, exactly:
// the normalised digit arrays to out_digits and / or the FP32 values to out, both in the order
// [p][q], or [q][p] with transpose (either may be null). nsm: SMs of the device.
cudaError_t launch_exact(const void* left, int ldl, const void* right, int ldr, bool dv, float alpha, int M, int P, int Q,
                         long long* part, bool transpose, long long* out_digits, float* out, int nsm, cudaStream_t st);
// n digit arrays: out_digits = normalised (a + b), out = the FP32 values (b, out_digits or out may be null)
cudaError_t launch_exact_combine(const long long* a, const long long* b, int64_t n, long long* out_digits, float* out,
                                 cudaStream_t st);
cudaError_t prepare_exact();
// Multiply-add rate probe of the exact mode (the roofline of its digit kernel): `products` is set
// to the number of 32-bit wide multiply-adds the launch performs; sink: exact_probe_sink_bytes.
size_t exact_probe_sink_bytes(int nsm);
cudaError_t launch_exact_rate_probe(int iters, long long* sink, int nsm, int64_t* products, cudaStream_t st);

// Raise the dynamic shared-memory limit of every kernel instance in a
// translation unit (once per device, with that device current).
cudaError_t prepare_down();
cudaError_t prepare_up();
cudaError_t prepare_wgrad();
cudaError_t prepare_dy();
cudaError_t prepare_dxda();

}  // namespace lora
