// common.cuh -- sm_103a building blocks shared by the LoRA delta kernels:
// mbarrier waits with a time limit, TMA tile copies, tcgen05 MMA / TMEM
// access, shared-memory matrix descriptors, and the fixed summation tree.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lora {

// ----------------------------------------------------------------- limits
// A wait on an mbarrier gives up after this long (ns of %globaltimer). Every
// wait covers one pipeline stage (or, in the cluster kernels, one peer's share
// of a tile, bounded on the host); the kernels finish in micro- to
// milliseconds, so reaching the limit means the pipeline is broken, and the
// kernel reports it and returns within a fraction of a second instead of
// holding the GPU.
constexpr uint64_t kWaitLimitNs = 100000000ull;    // 0.1 s
constexpr uint64_t kDrainLimitNs = 20000000ull;    // 0.02 s, for teardown waits

// Status block (the first bytes of the caller's workspace), 32-bit words:
//   word 0  status code, written by a kernel that gives up on a wait: (site << 8) | kDevTimeout;
//           only while the word is zero, so the first code (the root cause) stays
//   word 2  test hook: a kernel kind (kKindDown ...); the producer warp of that kernel first waits
//           on an mbarrier that nothing completes, so the wait runs out (0: off)
//   word 3  test hook: the wait limit in microseconds (0: kWaitLimitNs)
// Words 2 and 3 are read, never written, by the kernels.
constexpr uint32_t kDevTimeout = 1u;
constexpr uint32_t kKindDown = 1u, kKindUp = 2u, kKindDy = 3u, kKindWgrad = 4u;

// ------------------------------------------------------------ small utils
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }
__device__ __forceinline__ uint32_t warp_id() {
  return __shfl_sync(0xffffffffu, threadIdx.x >> 5, 0);
}

// --------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0u;
}

// Per-CTA abort state: a flag in shared memory, the caller's status word and the wait limit.
struct Abort {
  volatile uint32_t* flag;   // shared memory
  uint32_t* status;          // global (may be null)
  uint64_t limit_ns;         // a wait gives up after this long
};
// The abort state of a kernel: the wait limit is kWaitLimitNs unless word 3 of the status block
// overrides it (test hook). Call after the grid dependency wait.
__device__ __forceinline__ Abort make_abort(volatile uint32_t* flag, uint32_t* status) {
  const uint32_t us = status ? status[3] : 0u;
  return Abort{flag, status, us ? uint64_t(us) * 1000ull : kWaitLimitNs};
}
// True when word 2 of the status block asks this kind of kernel to stall (test hook).
__device__ __forceinline__ bool stall_requested(const uint32_t* status, uint32_t kind) {
  return status && status[2] == kind;
}

// Slow path of a bounded wait. Returns false when the CTA is aborting: either
// this wait ran past its limit (then it raises the abort flag and records
// `site` in the status word) or another thread of the CTA already did.
static __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, Abort ab, uint32_t site,
                                       uint64_t limit_ns, bool honour_abort) {
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test(bar, parity)) return true;
    if ((it & 31u) == 0u) {
      if (honour_abort && *ab.flag) return false;
      if (global_ns() - t0 > limit_ns) {
        *ab.flag = 1u;
        if (ab.status) atomicCAS(ab.status, 0u, (site << 8) | kDevTimeout);   // the first code stays
        return false;
      }
    }
  }
}

// Wait for the phase of `bar` with the given parity to complete, for at most
// the abort state's limit. False means "abort": skip the work, keep the control flow.
__device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, Abort ab, uint32_t site) {
  if (mbar_test(bar, parity)) return true;
  return wait_slow(bar, parity, ab, site, ab.limit_ns, true);
}
// The stall test hook: a wait on a barrier that nothing completes, given a quarter of the
// limit so that it runs out before any wait that depends on the stalled warp.
__device__ __forceinline__ void stall_wait(uint32_t never, Abort ab, uint32_t site) {
  wait_slow(never, 0u, ab, site, ab.limit_ns / 4, true);
}
// Teardown variant: ignores the abort flag, shorter limit.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, Abort ab, uint32_t site) {
  if (mbar_test(bar, parity)) return true;
  return wait_slow(bar, parity, ab, site, kDrainLimitNs, false);
}

// Pipeline ring position: stage index and the phase parity of that stage.
struct Ring {
  uint32_t idx = 0, phase = 0;
  template <int N>
  __device__ __forceinline__ void next() {
    if (++idx == N) { idx = 0; phase ^= 1u; }
  }
};

// ---------------------------------------------------------- thread-block clusters
// A cluster's CTAs run at the same time (the hardware schedules them together),
// so one may wait for another. Peers signal each other through mbarriers in the
// waiting CTA's shared memory (remote arrive, release at cluster scope; the
// waiter's try_wait acquires at cluster scope).
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster; orders shared and global memory at cluster scope.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The address of the same shared-memory location in the CTA of the given cluster rank.
__device__ __forceinline__ uint32_t peer_addr(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Arrive on an mbarrier of a peer CTA (address from peer_addr), releasing this thread's prior
// writes -- and those ordered before them by a CTA barrier -- at cluster scope.
__device__ __forceinline__ void mbar_arrive_peer(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_test_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0u;
}
// Bounded wait for a phase completed by cluster peers (acquire at cluster scope); false: abort.
static __device__ __noinline__ bool wait_cluster(uint32_t bar, uint32_t parity, Abort ab, uint32_t site) {
  if (mbar_test_cluster(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test_cluster(bar, parity)) return true;
    if ((it & 31u) == 0u) {
      if (*ab.flag) return false;
      if (global_ns() - t0 > ab.limit_ns) {
        *ab.flag = 1u;
        if (ab.status) atomicCAS(ab.status, 0u, (site << 8) | kDevTimeout);
        return false;
      }
    }
  }
}

// ------------------------------------------- programmatic dependent launch
// The kernels are launched with programmatic stream serialization: a kernel may
// start (barrier set-up, TMEM allocation, tensor-map prefetch) while its
// predecessor in the stream drains. Before touching global memory it waits for
// the predecessor to finish and its writes to be visible; right after, it lets
// its own successor start launching.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_map(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// Prefetch one tile of a tensor into L2 (no shared memory, no completion
// tracking). Issued before the grid dependency wait it warms L2 for the first
// loads after it while the predecessor drains; L2 is the point of coherence for
// those loads, so a line the predecessor writes meanwhile is read as written.
__device__ __forceinline__ void tma_prefetch_l2(const CUtensorMap* m, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(m)),
               "r"(x), "r"(y)
               : "memory");
}
// 2-D tiled load into shared memory; completes `bar`'s transaction count.
// x (innermost coordinate) must be a multiple of 16 bytes / element size.
__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap* m, uint32_t bar, int x, int y,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
// 2-D tiled store from shared memory (bulk-group completion), with an L2
// policy: the wide FP32 outputs are stored evict-first, so their lines leave
// L2 (are written back to HBM) while the storing kernel runs instead of being
// written back during the next kernel's read stream.
__device__ __forceinline__ void tma_store(const CUtensorMap* m, uint32_t src, int x, int y, uint64_t policy) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(src), "r"(x), "r"(y), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void tma_store_wait_all() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA / tensor core) reads of the same bytes.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Order generic-proxy global accesses (seen through an acquire) before later
// async-proxy (TMA) reads of global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void named_bar(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, BF16 inputs, FP32 accumulate. Issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// Load 8 consecutive 32-bit TMEM columns of this thread's lane (32x32b shape).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// Make later uses of loaded registers depend on the preceding tcgen05.wait::ld.
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (16-byte units), descriptor version 1, layout type.
constexpr uint32_t kLayoutNone = 0, kLayoutSW128 = 2, kLayoutSW64 = 4, kLayoutSW32 = 6;
__host__ __device__ constexpr uint32_t layout_for_span(int span_bytes) {
  return span_bytes == 128 ? kLayoutSW128 : (span_bytes == 64 ? kLayoutSW64 : kLayoutSW32);
}
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= static_cast<uint64_t>(layout) << 61;
  return d;
}
// The same descriptor `bytes` further on in shared memory. The start-address
// field holds address / 16 in 14 bits; every operand of these kernels lies
// below 256 KB, so the add never carries out of the field.
__device__ __forceinline__ uint64_t desc_advance(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

// One lane of a converged warp (the issuing thread of a tcgen05.mma / commit).
// Running the issue loop on the whole warp keeps its descriptor arithmetic
// warp-uniform, so it stays off the per-thread register path.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0u;
}

// Instruction descriptor, kind::f16: BF16 A and B, FP32 D, dense; a_mn / b_mn
// select MN-major (1) or K-major (0) operands.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ------------------------------------------------------------ arithmetic
// dV = bf16_rn(fp32(dY) * alpha) on 8 packed BF16 values (one 16-byte chunk).
__device__ __forceinline__ uint4 scale_bf16x8(uint4 v, float alpha) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(w[i] << 16);
    const float hi = __uint_as_float(w[i] & 0xFFFF0000u);
    const __nv_bfloat162 p = __floats2bfloat162_rn(__fmul_rn(lo, alpha), __fmul_rn(hi, alpha));
    w[i] = *reinterpret_cast<const uint32_t*>(&p);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// The same transform when alpha = 2^k (alpha > 0, |k| <= 12): the packed BF16
// multiply rounds the same exact product once, so it gives the same bits
// (zeros, subnormals, overflow to infinity and NaNs included: checked against
// the FP32 form above for all 65536 inputs and every such k) in a quarter of
// the instructions. pow2_bf16x2 returns alpha as BF16 in both halves of a
// word, or 0 when alpha is not of that form.
__device__ __forceinline__ uint32_t pow2_bf16x2(float alpha) {
  const uint32_t b = __float_as_uint(alpha);
  const uint32_t e = (b >> 23) & 0xFFu;
  if ((b & 0x807FFFFFu) != 0u || e < 127u - 12u || e > 127u + 12u) return 0u;
  return (b >> 16) * 0x00010001u;
}
__device__ __forceinline__ uint4 scale_bf16x8_pow2(uint4 v, uint32_t a2) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(w[i]) : "r"(w[i]), "r"(a2));
  return make_uint4(w[0], w[1], w[2], w[3]);
}
// alpha = 1: dV = bf16(fp32(dY) * 1) is dY itself for every BF16 value (a signaling NaN would
// only be quieted; the tensor core treats both as NaN), so the kernels pass dY through as dV
// without the shared-memory round trip of the transform.
__device__ __forceinline__ bool dv_is_dy(float alpha) { return alpha == 1.0f; }
// dV for one 16-byte chunk, taking the packed form when a2 != 0.
__device__ __forceinline__ uint4 dv_bf16x8(uint4 v, float alpha, uint32_t a2) {
  return a2 ? scale_bf16x8_pow2(v, a2) : scale_bf16x8(v, alpha);
}

// The fixed summation tree. Leaves are 16-term tensor-core dot products
// (fresh accumulator each), combined by the canonical pairwise tree over the
// leaf index: level l adds node i and node i + 2^l when i is a multiple of
// 2^(l+1) (a node with no partner passes up unchanged). Group of 4 leaves:
__device__ __forceinline__ float tree4(float l0, float l1, float l2, float l3) {
  return __fadd_rn(__fadd_rn(l0, l1), __fadd_rn(l2, l3));
}

// The canonical tree over 4 consecutive leaves of 8 columns each, read from TMEM starting at
// column `taddr`, leaves 16 columns apart (this warp's lane quarter): o[c] = tree4 of column c
// of the four leaves. !ok: no TMEM access, o = 0 (an aborting CTA).
__device__ __forceinline__ void leaves4_tree(uint32_t taddr, bool ok, float (&o)[8]) {
  uint32_t v[4][8];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 8; ++e) v[j][e] = 0u;
  if (ok) {
#pragma unroll
    for (int j = 0; j < 4; ++j) tmem_ld8(taddr + j * 16, v[j]);
    tmem_ld_wait();
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) reg_fence(v[j]);
#pragma unroll
  for (int c = 0; c < 8; ++c)
    o[c] = tree4(__uint_as_float(v[0][c]), __uint_as_float(v[1][c]), __uint_as_float(v[2][c]), __uint_as_float(v[3][c]));
}

// ------------------------------------------------ slice partials -> BF16 tile
// Canonical pairwise tree over the first n (<= NB, NB a power of two) of NB
// slices, for G groups of 8 consecutive FP32 values: group g of slice i is
// p[i * stride + 8 g .. 8 g + 7] (16-byte aligned). Slices past n are zero,
// which leaves every non-zero sum unchanged. All loads are issued before the
// first add (the partials were just written by the previous kernel: L2).
template <int NB, int G>
__device__ __forceinline__ void block_slices(const float* p, size_t stride, int n, float (&o)[G][8]) {
  float v[NB][G][8];
#pragma unroll
  for (int i = 0; i < NB; ++i)
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
      if (i < n) {
        const float4* q = reinterpret_cast<const float4*>(p + size_t(i) * stride + 8 * g);
        a = __ldcg(q);
        b = __ldcg(q + 1);
      }
      v[i][g][0] = a.x; v[i][g][1] = a.y; v[i][g][2] = a.z; v[i][g][3] = a.w;
      v[i][g][4] = b.x; v[i][g][5] = b.y; v[i][g][6] = b.z; v[i][g][7] = b.w;
    }
#pragma unroll
  for (int w = 1; w < NB; w <<= 1)
#pragma unroll
    for (int i = 0; i < NB; i += 2 * w)
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int c = 0; c < 8; ++c) v[i][g][c] = __fadd_rn(v[i][g][c], v[i + w][g][c]);
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int c = 0; c < 8; ++c) o[g][c] = v[0][g][c];
}

// Canonical pairwise tree over S slices (any S >= 1) of one group of 8 FP32
// values: blocks of 8 slices (above), then the canonical tree over the blocks.
__device__ __forceinline__ void sum_slices8(const float* p, size_t stride, int S, float (&o)[8]) {
  float (&o1)[1][8] = reinterpret_cast<float (&)[1][8]>(o);
  if (S <= 8) {
    block_slices<8, 1>(p, stride, S, o1);
    return;
  }
  float stk[24][8];
  int top = 0;
  for (int b = 0; b * 8 < S; ++b) {
    float x[1][8];
    block_slices<8, 1>(p + size_t(b) * 8 * stride, stride, min(8, S - 8 * b), x);
    for (int t = b; t & 1; t >>= 1) {
      --top;
#pragma unroll
      for (int c = 0; c < 8; ++c) x[0][c] = __fadd_rn(stk[top][c], x[0][c]);
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) stk[top][c] = x[0][c];
    ++top;
  }
  --top;
#pragma unroll
  for (int c = 0; c < 8; ++c) o[c] = stk[top][c];
  while (top > 0) {
    --top;
#pragma unroll
    for (int c = 0; c < 8; ++c) o[c] = __fadd_rn(stk[top][c], o[c]);
  }
}

// Round 8 FP32 values to BF16 (nearest even) and pack them into 16 bytes.
__device__ __forceinline__ uint4 pack_bf16x8(const float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 p2 = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&p2);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Canonical pairwise tree over the S slice partials (slice stride `stride`
// floats) of 8 consecutive FP32 values, rounded to BF16 and packed: the value
// of U (or dU) from the partial sums over slices of the reduction dimension.
// All loads of a block of slices are in flight together.
__device__ __forceinline__ uint4 slices_to_bf16x8(const float* p, size_t stride, int S) {
  float v[8];
  if (S <= 4) {
    float w[1][8];
    block_slices<4, 1>(p, stride, S, w);
#pragma unroll
    for (int c = 0; c < 8; ++c) v[c] = w[0][c];
  } else {
    sum_slices8(p, stride, S, v);
  }
  return pack_bf16x8(v);
}

// The same value for S > 8 slices, formed by four consecutive lanes of one warp (l4 = lane & 3,
// gmask = the four lanes' mask, all four active): lane l adds block 4 s + l of 8 slices (all its
// loads in flight; a partial last block is padded with zeros, as in the one-thread tree), the
// four block sums meet by shuffles in the canonical order (a block past the last one passes its
// partner up unchanged), and the sums of the 32-slice groups go through the canonical tree over
// the group index. Same bits as slices_to_bf16x8; every lane returns the packed value.
__device__ __forceinline__ uint4 slices_to_bf16x8_4lanes(const float* p, size_t stride, int S, int l4,
                                                         unsigned gmask) {
  const int nb = (S + 7) / 8, nsg = (nb + 3) / 4;
  float stk[24][8];
  int top = 0;
  for (int sg = 0; sg < nsg; ++sg) {
    const int b = 4 * sg + l4;
    float x[1][8];
    if (b < nb) {
      block_slices<8, 1>(p + size_t(b) * 8 * stride, stride, min(8, S - 8 * b), x);
    } else {
#pragma unroll
      for (int c = 0; c < 8; ++c) x[0][c] = 0.0f;
    }
    // pairs (0, 1) and (2, 3): left + right, or left alone when the right block does not exist
    const bool has_right = 4 * sg + (l4 | 1) < nb;
    float pr[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float y = __shfl_xor_sync(gmask, x[0][c], 1, 4);
      const float left = (l4 & 1) ? y : x[0][c], right = (l4 & 1) ? x[0][c] : y;
      pr[c] = has_right ? __fadd_rn(left, right) : left;
    }
    // the two pairs: (0, 1) + (2, 3), or (0, 1) alone when block 2 does not exist
    const bool has_second = 4 * sg + 2 < nb;
    float sgs[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float y = __shfl_xor_sync(gmask, pr[c], 2, 4);
      const float first = (l4 & 2) ? y : pr[c], second = (l4 & 2) ? pr[c] : y;
      sgs[c] = has_second ? __fadd_rn(first, second) : first;
    }
    // canonical tree over the 32-slice groups: merge once per trailing one of sg
    for (int t = sg; t & 1; t >>= 1) {
      --top;
#pragma unroll
      for (int c = 0; c < 8; ++c) sgs[c] = __fadd_rn(stk[top][c], sgs[c]);
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) stk[top][c] = sgs[c];
    ++top;
  }
  float o[8];
  --top;
#pragma unroll
  for (int c = 0; c < 8; ++c) o[c] = stk[top][c];
  while (top > 0) {
    --top;
#pragma unroll
    for (int c = 0; c < 8; ++c) o[c] = __fadd_rn(stk[top][c], o[c]);
  }
  return pack_bf16x8(o);
}

}  // namespace lora
