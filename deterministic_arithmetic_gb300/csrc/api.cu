// api.cu -- the C ABI (include/lora_delta.h): argument checks, TMA tensor
// maps, workspace carving and the launch sequence of the forward and backward
// passes. No allocation, no synchronisation on the compute path.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/lora_delta.h"
#include "kernels.h"

using namespace lora;

namespace {

constexpr size_t kStatusBytes = 256;
// Control block: the status block, then control words (the fused forward's tickets and row-tile
// words), zero before a workspace's first use and zero again after every call.
constexpr size_t kControlBytes = kStatusBytes + 65536;
static_assert(kControlBytes == LORA_DELTA_CONTROL_BYTES, "control block size of the public header");
static_assert(kFusedCtlWords * 4 <= 65536, "control words fit the control block");
constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool probed = false;
  bool usable = false;
  int num_sms = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

void* g_events[64];
int g_nevents = 0;

// Schedule of the single-site passes (lora_delta_set_schedule): separate launches, cluster
// reductions or single cluster launches; cluster size 0 = kDefaultCluster.
int g_schedule = LORA_SCHEDULE_AUTO;
int g_cluster = 0;
constexpr int kDefaultCluster = 4;
// A CTA of a cluster waits for its peers' share of a tile (forward: 128 rows x K / cl of x; backward:
// 256 rows x N / cl of dY): the cluster launches take shapes whose share is at most this many bytes
// (about a millisecond of streaming), far inside the kernels' wait limit; larger shapes run the
// separate launches.
constexpr int64_t kClusterShareBytes = int64_t(32) << 20;
int cluster_of_setting() { return g_cluster > 0 ? g_cluster : kDefaultCluster; }
int log2_cl(int cl) { return cl == 1 ? 0 : (cl == 2 ? 1 : (cl == 4 ? 2 : 3)); }
// Clusters of each instance that fit on a device at once: forward [device][RP 16 / 32][bf16 output]
// [with the expansion][log2 cl], backward [device][with phase C][log2 cl]; 0 = not yet queried.
int g_max_clusters[kMaxDevices][2][2][2][4];
int g_max_bwd_clusters[kMaxDevices][2][4];

// Clusters of cl CTAs of the forward cluster kernel instance that fit on the current device at
// once (queried once per device and instance); 0 when none.
int fwd_clusters(int RP, bool y_bf16, bool up, int cl) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  int& v = g_max_clusters[dev][RP == 16 ? 0 : 1][(y_bf16 && up) ? 1 : 0][up ? 1 : 0][log2_cl(cl)];
  if (v == 0) {
    int n = 0;
    if (fwd_cluster_max_clusters(RP, y_bf16 && up, up, cl, &n) != cudaSuccess || n < 1) return 0;
    v = n;
  }
  return v;
}

// The schedule a forward call of m active sites takes: the cluster schedules cover one site of
// padded rank 16 or 32 whose per-CTA share of a tile is small enough; automatic = separate (the
// cluster schedules measured no faster for the forward).
int fwd_schedule(int m, int RP, int64_t K) {
  const int sched = g_schedule == LORA_SCHEDULE_AUTO ? LORA_SCHEDULE_SEPARATE : g_schedule;
  if (m != 1 || RP > 32 || 128 * K * 2 / cluster_of_setting() > kClusterShareBytes) return LORA_SCHEDULE_SEPARATE;
  return sched;
}
// Rows per unit of the backward's cluster reductions: a 256-row chunk where the chunks give at
// least three quarters of the SMs a CTA, else one 128-row tile (twice the units).
int bwd_unit_rows(int64_t M, int cl, int nsm) {
  return 4 * ceil_div(M, kDyChunk) * cl >= 3 * int64_t(nsm) ? kDyChunk : 128;
}
// The schedule a backward call takes: one site of padded rank 16 with a small enough share;
// automatic = the cluster reductions where their 256-row chunks give at least three quarters of
// the SMs a CTA, else the separate launches (measured: with 128-row units, or fewer CTAs, the dY
// pass -- bound per SM -- on fewer SMs than the separate dy kernel's costs more than the rows
// launch it saves: fc1 78.7 vs 70.5 us).
int bwd_schedule(int m, int RP, int64_t M, int64_t N, int nsm) {
  const int cl = cluster_of_setting();
  if (m != 1 || RP != 16 || int64_t(kDyChunk) * N * 2 / cl > kClusterShareBytes) return LORA_SCHEDULE_SEPARATE;
  if (g_schedule != LORA_SCHEDULE_AUTO) return g_schedule;
  return bwd_unit_rows(M, cl, nsm) == kDyChunk ? LORA_SCHEDULE_CLUSTER_REDUCE : LORA_SCHEDULE_SEPARATE;
}

// The same for the backward cluster kernel.
int bwd_clusters(bool phase_c, int cl) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  int& v = g_max_bwd_clusters[dev][phase_c ? 1 : 0][log2_cl(cl)];
  if (v == 0) {
    int n = 0;
    if (bwd_cluster_max_clusters(phase_c, cl, &n) != cudaSuccess || n < 1) return 0;
    v = n;
  }
  return v;
}

lora_status device_ready(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LORA_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.probed) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return LORA_ERR_CUDA;
    d.probed = true;
    d.num_sms = sms;
    d.usable = (major == 10 && minor == 3);
    if (d.usable) {
      if (prepare_down() != cudaSuccess || prepare_up() != cudaSuccess || prepare_wgrad() != cudaSuccess ||
          prepare_dy() != cudaSuccess || prepare_exact() != cudaSuccess || prepare_fwd_fused() != cudaSuccess ||
          prepare_fwd_cluster() != cudaSuccess || prepare_bwd_cluster() != cudaSuccess || prepare_dxda() != cudaSuccess) {
        d.probed = false;
        return LORA_ERR_CUDA;
      }
    }
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn) {
        d.probed = false;
        return LORA_ERR_CUDA;
      }
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  if (!d.usable) return LORA_ERR_DEVICE;
  *num_sms = d.num_sms;
  return LORA_OK;
}

CUtensorMapSwizzle swizzle_for_span(int bytes) {
  return bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : (bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}

// 2-D row-major tensor [rows][cols] of `esize`-byte elements; box [box_rows][box_cols].
bool make_map(CUtensorMap* m, const void* ptr, bool f32, int64_t rows, int64_t cols, int box_cols, int box_rows,
              CUtensorMapSwizzle sw) {
  const CUtensorMapDataType dt = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t esize = f32 ? 4 : 2;
  cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(cols) * esize};
  cuuint32_t box[2] = {cuuint32_t(box_cols), cuuint32_t(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

lora_status check_shape(int64_t M, int64_t K, int64_t N, int64_t R) {
  if (M < 0 || K <= 0 || N <= 0 || (K % 8) != 0 || (N % 8) != 0) return LORA_ERR_SHAPE;
  if (M >= (int64_t(1) << 31) || K >= (int64_t(1) << 31) || N >= (int64_t(1) << 31)) return LORA_ERR_SHAPE;
  if (R < 8 || R > 64 || (R % 8) != 0) return LORA_ERR_RANK;
  return LORA_OK;
}

size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

// Scratch of one site (offsets from the start of the site's region; a call's workspace is the
// control block, then the regions of its sites in site order).
struct FwdLayout {
  size_t upart, bytes;     // U slice partials [S][M][RP]; region size
};
FwdLayout fwd_layout(int64_t M, int64_t K, int64_t R) {
  const int RP = padded_rank(int(R));
  const size_t S = size_t(ceil_div(K, down_slice(RP)));
  FwdLayout l;
  l.upart = 0;
  l.bytes = round256(S * size_t(M) * RP * 4);
  return l;
}
struct BwdLayout {
  size_t dupart, dbpart, dapart, bytes;   // dU slice partials, dB and dA chunk partials; region size
};
BwdLayout bwd_layout(int64_t M, int64_t K, int64_t N, int64_t R) {
  const int RP = padded_rank(int(R));
  const size_t S = size_t(ceil_div(N, du_slice(RP)));
  const size_t C = size_t(ceil_div(M, kWgradChunk));
  BwdLayout l;
  l.dupart = 0;
  l.dbpart = l.dupart + round256(S * size_t(M) * RP * 4);
  // dB partials per 128-row tile (the cluster reductions' units may be single tiles): up to 2 C
  l.dapart = l.dbpart + round256(size_t(ceil_div(M, 128)) * RP * size_t(N) * 4);
  l.bytes = l.dapart + round256(C * RP * size_t(K) * 4);
  return l;
}

struct Recorder {
  cudaStream_t st;
  int i = 0;
  explicit Recorder(cudaStream_t s) : st(s) {}
  void mark() {
    if (i < g_nevents && g_events[i]) cudaEventRecord(static_cast<cudaEvent_t>(g_events[i]), st);
    ++i;
  }
};

int grid_for(int64_t units, int nsm) { return int(std::max<int64_t>(1, std::min<int64_t>(units, nsm))); }

}  // namespace

extern "C" {

const char* lora_status_str(lora_status s) {
  switch (s) {
    case LORA_OK: return "ok";
    case LORA_ERR_NULL: return "a required pointer is NULL";
    case LORA_ERR_SHAPE: return "invalid shape (M >= 0; K, N positive multiples of 8; sizes below 2^31)";
    case LORA_ERR_ALIGN: return "a tensor or the workspace is not 16-byte aligned";
    case LORA_ERR_RANK: return "rank R must be a multiple of 8 in [8, 64]";
    case LORA_ERR_WORKSPACE: return "workspace too small";
    case LORA_ERR_CUDA: return "CUDA runtime or driver call failed";
    case LORA_ERR_DEVICE: return "current device is not an sm_103 (GB300) GPU";
    case LORA_ERR_TIMEOUT: return "a kernel gave up waiting (device status block)";
    default: return "unknown status";
  }
}

size_t lora_delta_fwd_workspace_size(int64_t M, int64_t K, int64_t N, int64_t R) {
  if (check_shape(M, K, N, R) != LORA_OK) return 0;
  return kControlBytes + fwd_layout(M, K, R).bytes;
}

size_t lora_delta_bwd_workspace_size(int64_t M, int64_t K, int64_t N, int64_t R) {
  if (check_shape(M, K, N, R) != LORA_OK) return 0;
  return kControlBytes + bwd_layout(M, K, N, R).bytes;
}

size_t lora_delta_fwd_workspace(int64_t M, int64_t K, int64_t N, int64_t R) {
  return lora_delta_fwd_workspace_size(M, K, N, R);
}

size_t lora_delta_bwd_workspace(int64_t M, int64_t K, int64_t N, int64_t R) {
  return lora_delta_bwd_workspace_size(M, K, N, R);
}

}  // extern "C"

namespace {

// One site of a call: the arguments of the single-site entry points, or one
// element of a grouped call.
struct FwdIn {
  const void *x, *a, *b;
  float alpha;
  int64_t M, K, N;
  void* delta_y;
  void* u;
};
struct BwdIn {
  const void *dy, *x, *a, *b, *u;
  float alpha;
  int64_t M, K, N;
  float *dx, *da, *db;
  void* du;
};

size_t fwd_site_bytes(int64_t M, int64_t K, int64_t R) { return fwd_layout(M, K, R).bytes; }
size_t bwd_site_bytes(int64_t M, int64_t K, int64_t N, int64_t R) { return bwd_layout(M, K, N, R).bytes; }

// Shared checks, in the order the single-site entry points document: shapes, NULL pointers,
// alignment, workspace size. *active = sites with M > 0 (indices), *need = workspace bytes.
template <class In, class Ptrs>
lora_status check_sites(const In* in, int n, int64_t R, const void* workspace, size_t workspace_bytes, Ptrs ptrs,
                        int* active, int* n_active) {
  if (n < 1 || n > kMaxSites) return LORA_ERR_SHAPE;
  for (int i = 0; i < n; ++i) {
    const lora_status s = check_shape(in[i].M, in[i].K, in[i].N, R);
    if (s != LORA_OK) return s;
  }
  *n_active = 0;
  for (int i = 0; i < n; ++i)
    if (in[i].M > 0) active[(*n_active)++] = i;
  if (*n_active == 0) return LORA_OK;
  for (int j = 0; j < *n_active; ++j)
    for (const void* p : ptrs(in[active[j]]))
      if (!p) return LORA_ERR_NULL;
  if (!workspace) return LORA_ERR_NULL;
  for (int j = 0; j < *n_active; ++j)
    for (const void* p : ptrs(in[active[j]]))
      if (!aligned16(p)) return LORA_ERR_ALIGN;
  if (!aligned16(workspace)) return LORA_ERR_ALIGN;
  return LORA_OK;
}

struct FwdPtrs {
  std::array<const void*, 5> operator()(const FwdIn& s) const { return {s.x, s.a, s.b, s.delta_y, s.u}; }
};
struct BwdPtrs {
  std::array<const void*, 9> operator()(const BwdIn& s) const {
    return {s.dy, s.x, s.a, s.b, s.u, s.dx, s.da, s.db, s.du};
  }
};

size_t fwd_need(const FwdIn* in, int n, int64_t R) {
  size_t t = kControlBytes;
  for (int i = 0; i < n; ++i)
    if (in[i].M > 0) t += fwd_site_bytes(in[i].M, in[i].K, R);
  return t;
}
size_t bwd_need(const BwdIn* in, int n, int64_t R) {
  size_t t = kControlBytes;
  for (int i = 0; i < n; ++i)
    if (in[i].M > 0) t += bwd_site_bytes(in[i].M, in[i].K, in[i].N, R);
  return t;
}

// The forward of every site: three launches over all sites' units (down, rows, up), or, with
// `fused` (one site, batches of up to kFusedMaxTiles row tiles), one launch doing the same
// three steps. Both give the same bits.
lora_status fwd_group(const FwdIn* in, int n, int64_t R, bool y_bf16, void* workspace, size_t workspace_bytes,
                      void* stream, bool fused = false) {
  int active[kMaxSites], m = 0;
  lora_status s = check_sites(in, n, R, workspace, workspace_bytes, FwdPtrs{}, active, &m);
  if (s != LORA_OK || m == 0) return s;
  if (workspace_bytes < fwd_need(in, n, R)) return LORA_ERR_WORKSPACE;
  int nsm = 0;
  if ((s = device_ready(&nsm)) != LORA_OK) return s;

  const int RP = padded_rank(int(R));
  const int span = RP * 2;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  DownArgs dargs{};
  RowsArgs rargs{};
  UpArgs uargs{};
  dargs.n = rargs.n = uargs.n = m;
  rargs.R = uargs.R = int(R);
  rargs.RP = RP;
  size_t off = kControlBytes;
  int64_t n_down = 0, n_up = 0;
  for (int j = 0; j < m; ++j) {
    const FwdIn& p = in[active[j]];
    const FwdLayout L = fwd_layout(p.M, p.K, R);
    float* upart = reinterpret_cast<float*>(ws + off + L.upart);
    off += L.bytes;
    DownSite& d = dargs.s[j];
    UpSite& q = uargs.s[j];
    if (!make_map(&d.in, p.x, false, p.M, p.K, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&d.w, p.a, false, R, p.K, 64, RP, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&q.a, p.u, false, p.M, R, RP, 128, swizzle_for_span(span)) ||
        !make_map(&q.b, p.b, false, p.N, R, RP, up_bn(RP), swizzle_for_span(span)) ||
        !(y_bf16 ? make_map(&q.out, p.delta_y, false, p.M, p.N, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B)
                 : make_map(&q.out, p.delta_y, true, p.M, p.N, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B)))
      return LORA_ERR_CUDA;
    d.part = upart;
    d.M = int(p.M);
    d.Kred = int(p.K);
    d.alpha = 1.0f;
    rargs.s[j] = RowsSite{upart, static_cast<__nv_bfloat16*>(p.u), int(p.M), int(ceil_div(p.K, down_slice(RP))), 0};
    q.M = int(p.M);
    q.Nout = int(p.N);
    q.alpha = p.alpha;
    n_down += down_units(p.M, p.K, RP);
    n_up += up_units(p.M, p.N, RP);
  }
  if (off > workspace_bytes) return LORA_ERR_WORKSPACE;   // every region inside the workspace
  Recorder rec(st);
  rec.mark();
  const int fcl = cluster_of_setting();
  const int sched = fused ? LORA_SCHEDULE_SEPARATE : fwd_schedule(m, RP, in[active[0]].K);
  if (sched != LORA_SCHEDULE_SEPARATE) {
    // single: one launch on clusters (down, rows and up steps per 128-row tile); reduce: the
    // down and rows steps on clusters, then the up-projection launch
    const bool single = sched == LORA_SCHEDULE_CLUSTER_SINGLE;
    const FwdIn& p = in[active[0]];
    const int mc = fwd_clusters(RP, y_bf16, single, fcl);
    if (mc < 1) return LORA_ERR_CUDA;
    FcArgs fa{};
    fa.x = dargs.s[0].in;
    fa.a = dargs.s[0].w;
    if (single) {
      fa.out = uargs.s[0].out;
      if (!make_map(&fa.b, p.b, false, p.N, R, RP, fc_bn(RP), swizzle_for_span(span))) return LORA_ERR_CUDA;
    }
    fa.part = dargs.s[0].part;
    fa.u = static_cast<__nv_bfloat16*>(p.u);
    fa.M = int(p.M);
    fa.K = int(p.K);
    fa.N = int(p.N);
    fa.R = int(R);
    fa.alpha = p.alpha;
    const int ncl = int(std::min<int64_t>(mc, ceil_div(p.M, 128)));
    if (launch_fwd_cluster(RP, y_bf16, single, fa, status, fcl, ncl, st) != cudaSuccess) return LORA_ERR_CUDA;
    rec.mark();
    if (!single) {
      if (launch_up(RP, false, y_bf16, uargs, status, grid_for(n_up, nsm), st) != cudaSuccess) return LORA_ERR_CUDA;
      rec.mark();
    }
    return LORA_OK;
  }
  if (fused && m == 1 && ceil_div(in[active[0]].M, 128) <= kFusedMaxTiles) {
    uint32_t* ctl = reinterpret_cast<uint32_t*>(ws + kStatusBytes);
    if (launch_fwd_fused(RP, y_bf16, dargs, uargs, static_cast<__nv_bfloat16*>(in[active[0]].u), int(R), ctl, nsm,
                         status, st) != cudaSuccess)
      return LORA_ERR_CUDA;
    rec.mark();
    return LORA_OK;
  }
  if (launch_down(RP, false, dargs, status, grid_for(n_down, nsm), st) != cudaSuccess) return LORA_ERR_CUDA;
  rec.mark();
  // U = bf16(tree over the K-slice partials), written to u
  if (launch_rows(rargs, nullptr, nsm, st) != cudaSuccess) return LORA_ERR_CUDA;
  rec.mark();
  if (launch_up(RP, false, y_bf16, uargs, status, grid_for(n_up, nsm), st) != cudaSuccess) return LORA_ERR_CUDA;
  rec.mark();
  return LORA_OK;
}

// The backward of every site: R <= 16: dy, dX (+ du), dA, combine; larger ranks: dU, dB, dX
// (+ du), dA, combine; each launch covers all sites' units.
lora_status bwd_group(const BwdIn* in, int n, int64_t R, void* workspace, size_t workspace_bytes, void* stream) {
  int active[kMaxSites], m = 0;
  lora_status s = check_sites(in, n, R, workspace, workspace_bytes, BwdPtrs{}, active, &m);
  if (s != LORA_OK || m == 0) return s;
  if (workspace_bytes < bwd_need(in, n, R)) return LORA_ERR_WORKSPACE;
  int nsm = 0;
  if ((s = device_ready(&nsm)) != LORA_OK) return s;

  const int RP = padded_rank(int(R));
  const int span = RP * 2;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  DyArgs yargs{};
  DownArgs dargs{};
  WgArgs bargs{}, aargs{};
  UpArgs uargs{};
  XaArgs xargs{};
  RowsArgs rargs{};
  CombineJobs da_jobs{}, db_jobs{};
  yargs.n = dargs.n = bargs.n = aargs.n = uargs.n = xargs.n = rargs.n = m;
  uargs.R = rargs.R = int(R);
  rargs.RP = RP;
  da_jobs.n = db_jobs.n = m;
  size_t off = kControlBytes;
  int64_t n_dy = 0, n_du = 0, n_db = 0, n_up = 0, n_da = 0, n_xa = 0;
  for (int j = 0; j < m; ++j) {
    const BwdIn& p = in[active[j]];
    const BwdLayout L = bwd_layout(p.M, p.K, p.N, R);
    float* dupart = reinterpret_cast<float*>(ws + off + L.dupart);
    float* dbpart = reinterpret_cast<float*>(ws + off + L.dbpart);
    float* dapart = reinterpret_cast<float*>(ws + off + L.dapart);
    off += L.bytes;
    const int M = int(p.M), K = int(p.K), N = int(p.N);
    const int C = int(ceil_div(p.M, kWgradChunk));
    UpSite& q = uargs.s[j];
    WgSite& wa = aargs.s[j];
    if (!make_map(&q.a, p.du, false, M, R, RP, 128, swizzle_for_span(span)) ||
        !make_map(&q.b, p.a, false, R, K, 64, RP, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&q.out, p.dx, true, M, K, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&wa.in, p.x, false, M, K, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&wa.g, p.du, false, M, R, RP, 64, swizzle_for_span(span)))
      return LORA_ERR_CUDA;
    if (RP == 16) {
      DySite& y = yargs.s[j];
      if (!make_map(&y.dy, p.dy, false, M, N, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
          !make_map(&y.b, p.b, false, N, R, RP, 128, swizzle_for_span(span)) ||
          !make_map(&y.u, p.u, false, M, R, RP, 128, swizzle_for_span(span)))
        return LORA_ERR_CUDA;
      y.du_part = dupart;
      y.db_part = dbpart;
      y.M = M;
      y.N = N;
      y.alpha = p.alpha;
      n_dy += ceil_div(M, kDyChunk) * ceil_div(N, kDySlice);
    } else {
      DownSite& d = dargs.s[j];
      WgSite& wb = bargs.s[j];
      if (!make_map(&d.in, p.dy, false, M, N, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
          !make_map(&d.w, p.b, false, N, R, RP, 64, swizzle_for_span(span)) ||
          !make_map(&wb.in, p.dy, false, M, N, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
          !make_map(&wb.g, p.u, false, M, R, RP, 64, swizzle_for_span(span)))
        return LORA_ERR_CUDA;
      d.part = dupart;
      d.M = M;
      d.Kred = N;
      d.alpha = p.alpha;
      wb.part = dbpart;
      wb.M = M;
      wb.Cw = N;
      wb.alpha = p.alpha;
      n_du += down_units(M, N, RP);
      n_db += wgrad_units(M, N, RP);
    }
    rargs.s[j] = RowsSite{dupart, static_cast<__nv_bfloat16*>(p.du), M, int(ceil_div(N, du_slice(RP))), 0};
    q.M = M;
    q.Nout = K;
    q.alpha = 1.0f;
    wa.part = dapart;
    wa.M = M;
    wa.Cw = K;
    wa.alpha = 1.0f;
    xargs.s[j] = XaSite{wa.in, q.b, q.a, q.out, dapart, M, K, 0, 0, 0};
    da_jobs.j[j] = CombineJob{dapart, p.da, C, K, int(R), RP, 0};
    db_jobs.j[j] = CombineJob{dbpart, p.db, C, N, int(R), RP, 1};
    n_up += up_units(M, K, RP);
    n_da += wgrad_units(M, K, RP);
    n_xa += dxda_units(M, K);
  }
  if (off > workspace_bytes) return LORA_ERR_WORKSPACE;   // every region inside the workspace
  Recorder rec(st);
  rec.mark();
  // dX and the dA chunk partials: one pass over x for padded rank 16, else the up-projection
  // and weight-gradient launches
  auto dx_da = [&]() -> bool {
    if (RP == 16) {
      if (launch_dxda(xargs, status, grid_for(n_xa, nsm), st) != cudaSuccess) return false;
      rec.mark();
      return true;
    }
    if (launch_up(RP, true, false, uargs, status, grid_for(n_up, nsm), st) != cudaSuccess) return false;
    rec.mark();
    if (launch_wgrad(RP, false, aargs, status, grid_for(n_da, nsm), st) != cudaSuccess) return false;
    rec.mark();
    return true;
  };
  const int bcl = cluster_of_setting();
  const int sched = bwd_schedule(m, RP, in[active[0]].M, in[active[0]].N, nsm);
  if (sched != LORA_SCHEDULE_SEPARATE) {
    // single: one launch on clusters (dU, dB partials; dU rows; dX, dA partials per 256-row chunk);
    // reduce: the dU, dB partials and dU rows on clusters, then the dX and dA launches. Then the
    // canonical trees over the chunk partials of dA and dB.
    const bool single = sched == LORA_SCHEDULE_CLUSTER_SINGLE;
    const BwdIn& p = in[active[0]];
    const int mc = bwd_clusters(single, bcl);
    if (mc < 1) return LORA_ERR_CUDA;
    BcArgs ba{};
    ba.dy = yargs.s[0].dy;
    ba.b = yargs.s[0].b;
    ba.u = yargs.s[0].u;
    if (single) {
      ba.x = aargs.s[0].in;
      ba.a = uargs.s[0].b;
      ba.dx = uargs.s[0].out;
    }
    ba.du_part = yargs.s[0].du_part;
    ba.db_part = yargs.s[0].db_part;
    ba.da_part = aargs.s[0].part;
    ba.du = static_cast<__nv_bfloat16*>(p.du);
    ba.M = int(p.M);
    ba.K = int(p.K);
    ba.N = int(p.N);
    ba.R = int(R);
    ba.alpha = p.alpha;
    ba.unit_rows = single ? kDyChunk : bwd_unit_rows(p.M, bcl, nsm);
    const int64_t n_units = ceil_div(p.M, ba.unit_rows);
    const int ncl = int(std::min<int64_t>(mc, n_units));
    if (launch_bwd_cluster(single, ba, status, bcl, ncl, st) != cudaSuccess) return LORA_ERR_CUDA;
    rec.mark();
    if (!single && !dx_da()) return LORA_ERR_CUDA;
    CombineJobs jobs{};
    jobs.n = 2;
    jobs.j[0] = da_jobs.j[0];
    jobs.j[1] = db_jobs.j[0];
    jobs.j[1].C = int(n_units);   // one dB partial per unit
    if (launch_combine(jobs, st) != cudaSuccess) return LORA_ERR_CUDA;
    rec.mark();
    return LORA_OK;
  }
  if (RP == 16) {
    // one pass over dY: dU partials over 512-column slices, dB partials over 256-row chunks
    if (launch_dy(yargs, status, grid_for(n_dy, nsm), st) != cudaSuccess) return LORA_ERR_CUDA;
    rec.mark();
  } else {
    // dU partials over slices of N (dV formed in shared memory)
    if (launch_down(RP, true, dargs, status, grid_for(n_du, nsm), st) != cudaSuccess) return LORA_ERR_CUDA;
    rec.mark();
    // dB chunk partials over 256-row chunks of M
    if (launch_wgrad(RP, true, bargs, status, grid_for(n_db, nsm), st) != cudaSuccess) return LORA_ERR_CUDA;
    rec.mark();
  }
  // dU = bf16(tree over the N-slice partials), written to du; in the same launch dB = the
  // canonical tree over the chunk partials just written (still in L2)
  if (launch_rows(rargs, &db_jobs, nsm, st) != cudaSuccess) return LORA_ERR_CUDA;
  rec.mark();
  if (!dx_da()) return LORA_ERR_CUDA;
  // dA: canonical tree over the chunk partials
  if (launch_combine(da_jobs, st) != cudaSuccess) return LORA_ERR_CUDA;
  rec.mark();
  return LORA_OK;
}
}  // namespace

extern "C" {

lora_status lora_delta_fwd(const void* x, const void* a, const void* b, float alpha, int64_t M, int64_t K, int64_t N,
                           int64_t R, float* delta_y, void* u, void* workspace, size_t workspace_bytes,
                           void* stream) {
  const FwdIn in{x, a, b, alpha, M, K, N, delta_y, u};
  return fwd_group(&in, 1, R, false, workspace, workspace_bytes, stream);
}

lora_status lora_delta_fwd_fused(const void* x, const void* a, const void* b, float alpha, int64_t M, int64_t K,
                                 int64_t N, int64_t R, void* delta_y, void* u, int y_bf16, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  const FwdIn in{x, a, b, alpha, M, K, N, delta_y, u};
  return fwd_group(&in, 1, R, y_bf16 != 0, workspace, workspace_bytes, stream, true);
}

lora_status lora_delta_fwd_bf16(const void* x, const void* a, const void* b, float alpha, int64_t M, int64_t K,
                                int64_t N, int64_t R, void* delta_y, void* u, void* workspace, size_t workspace_bytes,
                                void* stream) {
  const FwdIn in{x, a, b, alpha, M, K, N, delta_y, u};
  return fwd_group(&in, 1, R, true, workspace, workspace_bytes, stream);
}

lora_status lora_delta_bwd(const void* dy, const void* x, const void* a, const void* b, const void* u, float alpha,
                           int64_t M, int64_t K, int64_t N, int64_t R, float* dx, float* da, float* db, void* du,
                           void* workspace, size_t workspace_bytes, void* stream) {
  const BwdIn in{dy, x, a, b, u, alpha, M, K, N, dx, da, db, du};
  return bwd_group(&in, 1, R, workspace, workspace_bytes, stream);
}

size_t lora_delta_bwd_f32dy_workspace_size(int64_t M, int64_t K, int64_t N, int64_t R) {
  if (check_shape(M, K, N, R) != LORA_OK) return 0;
  return kControlBytes + bwd_layout(M, K, N, R).bytes + round256(size_t(M) * size_t(N) * 2);
}

lora_status lora_delta_bwd_f32dy(const float* dy, const void* x, const void* a, const void* b, const void* u,
                                 float alpha, int64_t M, int64_t K, int64_t N, int64_t R, float* dx, float* da,
                                 float* db, void* du, void* workspace, size_t workspace_bytes, void* stream) {
  lora_status s = check_shape(M, K, N, R);
  if (s != LORA_OK) return s;
  if (M == 0) return LORA_OK;
  if (!dy || !x || !a || !b || !u || !dx || !da || !db || !du || !workspace) return LORA_ERR_NULL;
  for (const void* p : {static_cast<const void*>(dy), x, a, b, u, static_cast<const void*>(dx),
                        static_cast<const void*>(da), static_cast<const void*>(db), static_cast<const void*>(du),
                        static_cast<const void*>(workspace)})
    if (!aligned16(p)) return LORA_ERR_ALIGN;
  const size_t bwd_bytes = kControlBytes + bwd_layout(M, K, N, R).bytes;
  if (workspace_bytes < lora_delta_bwd_f32dy_workspace_size(M, K, N, R)) return LORA_ERR_WORKSPACE;
  int nsm = 0;
  if ((s = device_ready(&nsm)) != LORA_OK) return s;
  // dV = bf16(fp32(dy * alpha)) into the workspace after the backward's own regions; the backward
  // then reads it as its dY with alpha = 1 (bf16(fp32(dv * 1)) = dv)
  void* dv = static_cast<uint8_t*>(workspace) + bwd_bytes;
  if (launch_dv_from_f32(dy, alpha, M * N, dv, nsm, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return LORA_ERR_CUDA;
  const BwdIn in{dv, x, a, b, u, 1.0f, M, K, N, dx, da, db, du};
  return bwd_group(&in, 1, R, workspace, bwd_bytes, stream);
}

size_t lora_delta_fwd_grouped_workspace_size(const lora_fwd_site* sites, int count, int64_t R) {
  if (!sites || count < 1 || count > kMaxSites) return 0;
  size_t t = kControlBytes;
  for (int i = 0; i < count; ++i) {
    if (check_shape(sites[i].M, sites[i].K, sites[i].N, R) != LORA_OK) return 0;
    t += fwd_site_bytes(sites[i].M, sites[i].K, R);
  }
  return t;
}

size_t lora_delta_bwd_grouped_workspace_size(const lora_bwd_site* sites, int count, int64_t R) {
  if (!sites || count < 1 || count > kMaxSites) return 0;
  size_t t = kControlBytes;
  for (int i = 0; i < count; ++i) {
    if (check_shape(sites[i].M, sites[i].K, sites[i].N, R) != LORA_OK) return 0;
    t += bwd_site_bytes(sites[i].M, sites[i].K, sites[i].N, R);
  }
  return t;
}

lora_status lora_delta_fwd_grouped(const lora_fwd_site* sites, int count, int64_t R, int y_bf16, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  if (!sites) return LORA_ERR_NULL;
  if (count < 1 || count > kMaxSites) return LORA_ERR_SHAPE;
  FwdIn in[kMaxSites];
  for (int i = 0; i < count; ++i)
    in[i] = FwdIn{sites[i].x, sites[i].a, sites[i].b, sites[i].alpha, sites[i].M, sites[i].K, sites[i].N,
                  sites[i].delta_y, sites[i].u};
  return fwd_group(in, count, R, y_bf16 != 0, workspace, workspace_bytes, stream);
}

lora_status lora_delta_bwd_grouped(const lora_bwd_site* sites, int count, int64_t R, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  if (!sites) return LORA_ERR_NULL;
  if (count < 1 || count > kMaxSites) return LORA_ERR_SHAPE;
  BwdIn in[kMaxSites];
  for (int i = 0; i < count; ++i)
    in[i] = BwdIn{sites[i].dy, sites[i].x, sites[i].a, sites[i].b, sites[i].u, sites[i].alpha, sites[i].M,
                  sites[i].K, sites[i].N, sites[i].dx, sites[i].da, sites[i].db, sites[i].du};
  return bwd_group(in, count, R, workspace, workspace_bytes, stream);
}

int lora_delta_exact_slots(void) { return kExactSlots; }

size_t lora_delta_grads_exact_workspace_size(int64_t M, int64_t K, int64_t N, int64_t R) {
  if (check_shape(M, K, N, R) != LORA_OK || M >= (int64_t(1) << 30) || R * K >= (int64_t(1) << 31) ||
      R * N >= (int64_t(1) << 31))
    return 0;
  return round256(std::max(exact_part_bytes(M, R, K), exact_part_bytes(M, R, N)));
}

lora_status lora_delta_grads_exact(const void* dy, const void* x, const void* u, const void* du, float alpha,
                                   int64_t M, int64_t K, int64_t N, int64_t R, float* da, float* db,
                                   int64_t* da_digits, int64_t* db_digits, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  lora_status s = check_shape(M, K, N, R);
  if (s != LORA_OK) return s;
  if (M >= (int64_t(1) << 30) || R * K >= (int64_t(1) << 31) || R * N >= (int64_t(1) << 31)) return LORA_ERR_SHAPE;
  const bool want_a = da || da_digits, want_b = db || db_digits;
  if (!want_a && !want_b) return LORA_OK;
  // inputs are read only when M > 0 (an empty batch gives zero gradients)
  if (!workspace || (M > 0 && ((want_a && (!x || !du)) || (want_b && (!dy || !u))))) return LORA_ERR_NULL;
  for (const void* p : {dy, x, u, du, static_cast<const void*>(da), static_cast<const void*>(db),
                        static_cast<const void*>(da_digits), static_cast<const void*>(db_digits),
                        static_cast<const void*>(workspace)})
    if (p && !aligned16(p)) return LORA_ERR_ALIGN;
  if (workspace_bytes < lora_delta_grads_exact_workspace_size(M, K, N, R)) return LORA_ERR_WORKSPACE;
  int nsm = 0;
  if ((s = device_ready(&nsm)) != LORA_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  long long* part = static_cast<long long*>(workspace);
  Recorder rec(st);
  rec.mark();
  // dA = du^T x: left du [M][R], right x [M][K], out [R][K]
  if (want_a && launch_exact(du, int(R), x, int(K), false, 1.0f, int(M), int(R), int(K), part, false,
                             reinterpret_cast<long long*>(da_digits), da, nsm, st) != cudaSuccess)
    return LORA_ERR_CUDA;
  rec.mark();
  // dB = dv^T u: left u [M][R], right dv from dy [M][N], out transposed to [N][R]
  if (want_b && launch_exact(u, int(R), dy, int(N), true, alpha, int(M), int(R), int(N), part, true,
                             reinterpret_cast<long long*>(db_digits), db, nsm, st) != cudaSuccess)
    return LORA_ERR_CUDA;
  rec.mark();
  return LORA_OK;
}

size_t lora_delta_grads_exact_f32dy_workspace_size(int64_t M, int64_t K, int64_t N, int64_t R) {
  const size_t e = lora_delta_grads_exact_workspace_size(M, K, N, R);
  return e ? e + round256(size_t(M) * size_t(N) * 2) : 0;
}

lora_status lora_delta_grads_exact_f32dy(const float* dy, const void* x, const void* u, const void* du, float alpha,
                                         int64_t M, int64_t K, int64_t N, int64_t R, float* da, float* db,
                                         int64_t* da_digits, int64_t* db_digits, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  lora_status s = check_shape(M, K, N, R);
  if (s != LORA_OK) return s;
  const size_t exact_bytes = lora_delta_grads_exact_workspace_size(M, K, N, R);
  if (!exact_bytes) return LORA_ERR_SHAPE;
  const bool want_b = db || db_digits;
  if (!workspace) return LORA_ERR_NULL;
  if (M > 0 && want_b && !dy) return LORA_ERR_NULL;
  if ((dy && !aligned16(dy)) || !aligned16(workspace)) return LORA_ERR_ALIGN;
  if (workspace_bytes < lora_delta_grads_exact_f32dy_workspace_size(M, K, N, R)) return LORA_ERR_WORKSPACE;
  // dV = bf16(fp32(dy * alpha)) into the workspace after the digit kernel's scratch; the exact
  // pass then reads it as its dY with alpha = 1 (bf16(fp32(dv * 1)) = dv)
  void* dv = static_cast<uint8_t*>(workspace) + exact_bytes;
  if (M > 0 && want_b) {
    int nsm = 0;
    if ((s = device_ready(&nsm)) != LORA_OK) return s;
    if (launch_dv_from_f32(dy, alpha, M * N, dv, nsm, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return LORA_ERR_CUDA;
  }
  return lora_delta_grads_exact(want_b ? dv : nullptr, x, u, du, 1.0f, M, K, N, R, da, db, da_digits, db_digits,
                                workspace, exact_bytes, stream);
}

lora_status lora_delta_exact_rate_probe(int64_t iters, void* sink, size_t sink_bytes, int64_t* products,
                                        void* stream) {
  if (!products) return LORA_ERR_NULL;
  if (iters < 1 || iters >= (int64_t(1) << 31)) return LORA_ERR_SHAPE;
  int nsm = 0;
  lora_status s = device_ready(&nsm);
  if (s != LORA_OK) return s;
  if (!sink) return LORA_ERR_NULL;
  if (!aligned16(sink)) return LORA_ERR_ALIGN;
  if (sink_bytes < exact_probe_sink_bytes(nsm)) return LORA_ERR_WORKSPACE;
  return launch_exact_rate_probe(int(iters), static_cast<long long*>(sink), nsm, products,
                                 static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

size_t lora_delta_exact_rate_probe_sink_bytes(void) {
  int nsm = 0;
  if (device_ready(&nsm) != LORA_OK) return 0;
  return exact_probe_sink_bytes(nsm);
}

lora_status lora_delta_exact_combine(const int64_t* a, const int64_t* b, int64_t n, int64_t* out_digits, void* stream) {
  if (n < 0 || n >= (int64_t(1) << 38)) return LORA_ERR_SHAPE;   // grid of n / 256 blocks
  if (n == 0) return LORA_OK;
  if (!a || !out_digits) return LORA_ERR_NULL;
  int nsm = 0;
  lora_status s = device_ready(&nsm);
  if (s != LORA_OK) return s;
  return launch_exact_combine(reinterpret_cast<const long long*>(a), reinterpret_cast<const long long*>(b), n,
                              reinterpret_cast<long long*>(out_digits), nullptr,
                              static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

lora_status lora_delta_exact_finalize(const int64_t* digits, int64_t n, float* out, void* stream) {
  if (n < 0 || n >= (int64_t(1) << 38)) return LORA_ERR_SHAPE;   // grid of n / 256 blocks
  if (n == 0) return LORA_OK;
  if (!digits || !out) return LORA_ERR_NULL;
  int nsm = 0;
  lora_status s = device_ready(&nsm);
  if (s != LORA_OK) return s;
  return launch_exact_combine(reinterpret_cast<const long long*>(digits), nullptr, n, nullptr, out,
                              static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? LORA_OK
             : LORA_ERR_CUDA;
}

lora_status lora_delta_device_status(const void* workspace, int* code) {
  if (!workspace || !code) return LORA_ERR_NULL;
  uint32_t v = 0;
  if (cudaMemcpy(&v, workspace, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return LORA_ERR_CUDA;
  *code = int(v);
  return v == 0 ? LORA_OK : LORA_ERR_TIMEOUT;
}

lora_status lora_delta_set_schedule(int schedule, int cluster_size) {
  if (schedule != LORA_SCHEDULE_SEPARATE && schedule != LORA_SCHEDULE_CLUSTER_REDUCE &&
      schedule != LORA_SCHEDULE_CLUSTER_SINGLE && schedule != LORA_SCHEDULE_AUTO)
    return LORA_ERR_SHAPE;
  if (cluster_size != 0 && cluster_size != 2 && cluster_size != 4 && cluster_size != 8) return LORA_ERR_SHAPE;
  g_schedule = schedule;
  g_cluster = cluster_size;
  return LORA_OK;
}

int lora_delta_schedule(int* cluster_size) {
  if (cluster_size) *cluster_size = g_cluster;
  return g_schedule;
}

lora_status lora_delta_plan(int backward, int64_t M, int64_t K, int64_t N, int64_t R, int* schedule, int* launches) {
  if (!schedule || !launches) return LORA_ERR_NULL;
  const lora_status s0 = check_shape(M, K, N, R);
  if (s0 != LORA_OK) return s0;
  int nsm = 0;
  const lora_status s1 = device_ready(&nsm);
  if (s1 != LORA_OK) return s1;
  const int RP = padded_rank(int(R));
  if (M == 0) {
    *schedule = LORA_SCHEDULE_SEPARATE;
    *launches = 0;
    return LORA_OK;
  }
  if (!backward) {
    const int sc = fwd_schedule(1, RP, K);
    *schedule = sc;
    *launches = sc == LORA_SCHEDULE_CLUSTER_SINGLE ? 1 : (sc == LORA_SCHEDULE_CLUSTER_REDUCE ? 2 : 3);
  } else {
    const int sc = bwd_schedule(1, RP, M, N, nsm);
    *schedule = sc;
    // padded rank 16: dX and dA in one launch (cluster reductions: dy + rows, dX + dA, combine;
    // separate: dy, rows, dX + dA, combine); above: dU, dB, rows, dX, dA, combine
    *launches = sc == LORA_SCHEDULE_CLUSTER_SINGLE ? 2 : (sc == LORA_SCHEDULE_CLUSTER_REDUCE ? 3 : (RP == 16 ? 4 : 6));
  }
  return LORA_OK;
}

lora_status lora_delta_set_profile_events(void* const* events, int count) {
  if (count < 0 || count > 64) return LORA_ERR_SHAPE;
  if (count > 0 && !events) return LORA_ERR_NULL;
  for (int i = 0; i < count; ++i) g_events[i] = events[i];
  g_nevents = count;
  return LORA_OK;
}

size_t lora_delta_describe(char* buf, size_t len) {
  char tmp[1024];
  const int n = std::snprintf(
      tmp, sizeof tmp,
      "{\"operator\": \"shared LoRA delta, forward + backward\", "
      "\"numeric_profile\": \"bf16 inputs; 16-term tcgen05 leaves (fresh FP32 accumulator); "
      "canonical pairwise FP32 tree over leaves; BF16 rounding of U, dV, dU\", "
      "\"reduction\": \"tree depends only on the reduction length; K-slices %d/%d/%d (R<=16/32/64), "
      "batch chunks %d rows; R<=16 backward reads dY once for dU (512-column slices) and dB; "
      "no split-K on M, no atomics\", "
      "\"tiles\": \"down 128x64 stages, up 128x(256/(RP/16)), wgrad 128 cols x 64 rows\", "
      "\"arch\": \"sm_103a\"}",
      down_slice(16), down_slice(32), down_slice(64), kWgradChunk);
  const size_t need = size_t(n) + 1;
  if (buf && len) {
    const size_t c = std::min(len - 1, size_t(n));
    std::memcpy(buf, tmp, c);
    buf[c] = '\0';
  }
  return need;
}

}  // extern "C"
