// api.cu -- the C ABI (include/lora_delta.h): argument checks, TMA tensor
// maps, workspace carving and the launch sequence of the forward and backward
// passes. No allocation, no synchronisation on the compute path.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/lora_delta.h"
#include "kernels.h"

using namespace lora;

namespace {

constexpr size_t kStatusBytes = 256;
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
          prepare_dy() != cudaSuccess) {
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

struct FwdLayout {
  size_t upart, total;
};
FwdLayout fwd_layout(int64_t M, int64_t K, int64_t R) {
  const int RP = padded_rank(int(R));
  const size_t S = size_t(ceil_div(K, down_slice(RP)));
  FwdLayout l;
  l.upart = kStatusBytes;
  l.total = l.upart + round256(S * size_t(M) * RP * 4);
  return l;
}
struct BwdLayout {
  size_t dupart, dbpart, dapart, total;
};
BwdLayout bwd_layout(int64_t M, int64_t K, int64_t N, int64_t R) {
  const int RP = padded_rank(int(R));
  const size_t S = size_t(ceil_div(N, du_slice(RP)));
  const size_t C = size_t(ceil_div(M, kWgradChunk));
  BwdLayout l;
  l.dupart = kStatusBytes;
  l.dbpart = l.dupart + round256(S * size_t(M) * RP * 4);
  l.dapart = l.dbpart + round256(C * RP * size_t(N) * 4);
  l.total = l.dapart + round256(C * RP * size_t(K) * 4);
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

const char* lora_status_str(int s) {
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
  return fwd_layout(M, K, R).total;
}

size_t lora_delta_bwd_workspace_size(int64_t M, int64_t K, int64_t N, int64_t R) {
  if (check_shape(M, K, N, R) != LORA_OK) return 0;
  return bwd_layout(M, K, N, R).total;
}

namespace {
lora_status fwd_impl(const void* x, const void* a, const void* b, float alpha, int64_t M, int64_t K, int64_t N,
                     int64_t R, void* delta_y, bool y_bf16, void* u, void* workspace, size_t workspace_bytes,
                     void* stream) {
  lora_status s = check_shape(M, K, N, R);
  if (s != LORA_OK) return s;
  if (M == 0) return LORA_OK;
  if (!x || !a || !b || !delta_y || !u || !workspace) return LORA_ERR_NULL;
  if (!aligned16(x) || !aligned16(a) || !aligned16(b) || !aligned16(delta_y) || !aligned16(u) || !aligned16(workspace))
    return LORA_ERR_ALIGN;
  const FwdLayout L = fwd_layout(M, K, R);
  if (workspace_bytes < L.total) return LORA_ERR_WORKSPACE;
  int nsm = 0;
  if ((s = device_ready(&nsm)) != LORA_OK) return s;

  const int RP = padded_rank(int(R));
  const int span = RP * 2;
  CUtensorMap m_x, m_a, m_b, m_y, m_u;
  if (!make_map(&m_x, x, false, M, K, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map(&m_u, u, false, M, R, RP, 128, swizzle_for_span(span)) ||
      !make_map(&m_a, a, false, R, K, 64, RP, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&m_b, b, false, N, R, RP, up_bn(RP), swizzle_for_span(span)) ||
      !(y_bf16 ? make_map(&m_y, delta_y, false, M, N, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B)
              : make_map(&m_y, delta_y, true, M, N, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B)))
    return LORA_ERR_CUDA;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  float* upart = reinterpret_cast<float*>(ws + L.upart);
  Recorder rec(st);
  rec.mark();
  if (launch_down(RP, false, m_x, m_a, upart, int(M), int(K), 1.0f, status, grid_for(down_units(M, K, RP), nsm), st) !=
      cudaSuccess)
    return LORA_ERR_CUDA;
  rec.mark();
  // U = bf16(tree over the K-slice partials), built inside the up-projection, which also writes u
  if (launch_up(RP, false, y_bf16, m_u, m_b, m_y, upart, int(ceil_div(K, down_slice(RP))), u, int(R), int(M), int(N),
                alpha, status, grid_for(up_units(M, N, RP), nsm), st) != cudaSuccess)
    return LORA_ERR_CUDA;
  rec.mark();
  return LORA_OK;
}
}  // namespace

lora_status lora_delta_fwd(const void* x, const void* a, const void* b, float alpha, int64_t M, int64_t K, int64_t N,
                           int64_t R, float* delta_y, void* u, void* workspace, size_t workspace_bytes,
                           void* stream) {
  return fwd_impl(x, a, b, alpha, M, K, N, R, delta_y, false, u, workspace, workspace_bytes, stream);
}

lora_status lora_delta_fwd_bf16(const void* x, const void* a, const void* b, float alpha, int64_t M, int64_t K,
                                int64_t N, int64_t R, void* delta_y, void* u, void* workspace, size_t workspace_bytes,
                                void* stream) {
  return fwd_impl(x, a, b, alpha, M, K, N, R, delta_y, true, u, workspace, workspace_bytes, stream);
}

lora_status lora_delta_bwd(const void* dy, const void* x, const void* a, const void* b, const void* u, float alpha,
                           int64_t M, int64_t K, int64_t N, int64_t R, float* dx, float* da, float* db, void* du,
                           void* workspace, size_t workspace_bytes, void* stream) {
  lora_status s = check_shape(M, K, N, R);
  if (s != LORA_OK) return s;
  if (M == 0) return LORA_OK;
  if (!dy || !x || !a || !b || !u || !dx || !da || !db || !du || !workspace) return LORA_ERR_NULL;
  for (const void* p : {dy, x, a, b, u, static_cast<const void*>(dx), static_cast<const void*>(da),
                        static_cast<const void*>(db), static_cast<const void*>(du), static_cast<const void*>(workspace)})
    if (!aligned16(p)) return LORA_ERR_ALIGN;
  const BwdLayout L = bwd_layout(M, K, N, R);
  if (workspace_bytes < L.total) return LORA_ERR_WORKSPACE;
  int nsm = 0;
  if ((s = device_ready(&nsm)) != LORA_OK) return s;

  const int RP = padded_rank(int(R));
  const int span = RP * 2;
  CUtensorMap m_dy_rows, m_b_rows, m_dy_chunk, m_u_chunk, m_a, m_dx, m_x_chunk, m_du_chunk, m_b_128, m_u_128, m_du_128;
  if (!make_map(&m_dy_rows, dy, false, M, N, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map(&m_b_rows, b, false, N, R, RP, 64, swizzle_for_span(span)) ||
      !make_map(&m_dy_chunk, dy, false, M, N, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&m_u_chunk, u, false, M, R, RP, 64, swizzle_for_span(span)) ||
      !make_map(&m_a, a, false, R, K, 64, RP, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&m_dx, dx, true, M, K, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&m_x_chunk, x, false, M, K, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&m_du_chunk, du, false, M, R, RP, 64, swizzle_for_span(span)) ||
      !make_map(&m_b_128, b, false, N, R, RP, 128, swizzle_for_span(span)) ||
      !make_map(&m_u_128, u, false, M, R, RP, 128, swizzle_for_span(span)) ||
      !make_map(&m_du_128, du, false, M, R, RP, 128, swizzle_for_span(span)))
    return LORA_ERR_CUDA;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  float* dupart = reinterpret_cast<float*>(ws + L.dupart);
  float* dbpart = reinterpret_cast<float*>(ws + L.dbpart);
  float* dapart = reinterpret_cast<float*>(ws + L.dapart);
  const int S = int(ceil_div(N, du_slice(RP)));
  const int C = int(ceil_div(M, kWgradChunk));
  Recorder rec(st);
  rec.mark();
  if (RP == 16) {
    // one pass over dY: dU partials over 512-column slices, dB partials over 256-row chunks
    if (launch_dy(m_dy_rows, m_b_128, m_u_128, dupart, dbpart, int(M), int(N), alpha, status,
                  grid_for(ceil_div(M, kDyChunk) * ceil_div(N, kDySlice), nsm), st) != cudaSuccess)
      return LORA_ERR_CUDA;
    rec.mark();
  } else {
    // dU partials over slices of N (dV formed in shared memory)
    if (launch_down(RP, true, m_dy_rows, m_b_rows, dupart, int(M), int(N), alpha, status,
                    grid_for(down_units(M, N, RP), nsm), st) != cudaSuccess)
      return LORA_ERR_CUDA;
    rec.mark();
    // dB chunk partials over 256-row chunks of M
    if (launch_wgrad(RP, true, m_dy_chunk, m_u_chunk, dbpart, int(M), int(N), alpha, status,
                     grid_for(wgrad_units(M, N, RP), nsm), st) != cudaSuccess)
      return LORA_ERR_CUDA;
    rec.mark();
  }
  // dU = bf16(tree over the N-slice partials), built inside the dX expansion, which also writes du
  if (launch_up(RP, true, false, m_du_128, m_a, m_dx, dupart, S, du, int(R), int(M), int(K), 1.0f, status,
                grid_for(up_units(M, K, RP), nsm), st) != cudaSuccess)
    return LORA_ERR_CUDA;
  rec.mark();
  if (launch_wgrad(RP, false, m_x_chunk, m_du_chunk, dapart, int(M), int(K), 1.0f, status,
                   grid_for(wgrad_units(M, K, RP), nsm), st) != cudaSuccess)
    return LORA_ERR_CUDA;
  rec.mark();
  // dA and dB: canonical tree over the chunk partials
  CombineJob jobs[2] = {{dapart, da, C, int(K), int(R), RP, 0}, {dbpart, db, C, int(N), int(R), RP, 1}};
  if (launch_combine(jobs, 2, st) != cudaSuccess) return LORA_ERR_CUDA;
  rec.mark();
  return LORA_OK;
}

lora_status lora_delta_device_status(const void* workspace, int* code) {
  if (!workspace || !code) return LORA_ERR_NULL;
  uint32_t v = 0;
  if (cudaMemcpy(&v, workspace, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return LORA_ERR_CUDA;
  *code = int(v);
  return v == 0 ? LORA_OK : LORA_ERR_TIMEOUT;
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
