// sched.cuh -- how the work units of a kernel phase reach its warp roles.
//
// Every role of a persistent CTA (TMA producer, MMA issuer, epilogue, ...)
// walks the same sequence of units. Two ways to make that sequence:
//
//   StaticSched  round robin: unit blockIdx.x, then + gridDim.x. No CTA ever
//                depends on another, so a plain launch is enough.
//   QueueSched   units claimed at run time from a global ticket counter by the
//                producer and handed to the other roles through a small ring
//                in shared memory. A unit is only ever claimed by a CTA that is
//                running, so a CTA may wait for a unit another CTA has claimed
//                (it will be finished) without any assumption about which CTAs
//                are resident: dependent phases of one launch need no
//                cooperative launch and no grid-wide barrier.
//
// Both present one interface: first() and next(u) give the role's units in
// order, -1 at the end.
#pragma once

#include "common.cuh"

namespace lora {

struct StaticSched {
  int total;
  __device__ __forceinline__ int first() const { return int(blockIdx.x) < total ? int(blockIdx.x) : -1; }
  __device__ __forceinline__ int next(int u) const {
    u += int(gridDim.x);
    return u < total ? u : -1;
  }
};

// The shared-memory ring of a QueueSched: kQ slots of a unit index, a `full`
// mbarrier per slot (one arrival: the producer publishing it) and a `free`
// mbarrier per slot (one arrival per reader warp when it moves on).
constexpr int kQueueSlots = 4;
struct QueueRing {
  volatile int* id;        // [kQueueSlots] unit indices (-1: no more units)
  uint32_t full0, free0;   // mbarrier addresses of slot 0 (8 bytes apart)
  __device__ __forceinline__ uint32_t full(int s) const { return full0 + 8u * s; }
  __device__ __forceinline__ uint32_t free_(int s) const { return free0 + 8u * s; }
  // thread 0, before the kernel's mbarrier init fence: `readers` = reader warps per slot
  __device__ __forceinline__ void init(int readers) const {
    for (int s = 0; s < kQueueSlots; ++s) {
      mbar_init(full(s), 1);
      mbar_init(free_(s), readers);
    }
  }
};

// Producer side (one thread): claims tickets from *counter (tickets below n are units) and
// publishes them. The next ticket is requested one unit ahead, so its latency overlaps the work.
struct QueueProducer {
  QueueRing q;
  unsigned int* counter;
  int n;
  Abort ab;
  uint32_t site;
  int k = 0;
  int pending = -1;
  __device__ __forceinline__ int publish(int u) {
    const int s = k % kQueueSlots;
    const bool ok = wait(q.free_(s), ((k / kQueueSlots) & 1) ^ 1u, ab, site);
    if (!ok) u = -1;                                     // aborting: end the sequence
    q.id[s] = u;
    mbar_arrive(q.full(s));                              // release: the index before the arrival
    ++k;
    return u;
  }
  __device__ __forceinline__ int claim() {
    const int t = pending < 0 ? int(atomicAdd(counter, 1u)) : pending;
    pending = t < n ? int(atomicAdd(counter, 1u)) : n;   // the following ticket, in flight meanwhile
    return t < n ? t : -1;
  }
  __device__ __forceinline__ int first() { return publish(claim()); }
  __device__ __forceinline__ int next(int) { return publish(claim()); }
};

// Reader side (one warp, all lanes call it; lane 0 arrives for the warp).
struct QueueReader {
  QueueRing q;
  Abort ab;
  uint32_t site;
  int k = 0;
  __device__ __forceinline__ int take() {
    const int s = k % kQueueSlots;
    const bool ok = __all_sync(0xffffffffu, wait(q.full(s), (k / kQueueSlots) & 1, ab, site));
    const int u = ok ? q.id[s] : -1;
    ++k;
    return u;
  }
  __device__ __forceinline__ int first() { return take(); }
  __device__ __forceinline__ int next(int) {
    __syncwarp();
    if ((threadIdx.x & 31u) == 0u) mbar_arrive(q.free_((k - 1) % kQueueSlots));   // done with the previous unit
    return take();
  }
};

// ------------------------------------------------------------ global flags
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Wait (one thread) until *p >= target, for at most the abort state's limit; false means abort
// (the limit ran out here, or another role of the CTA raised the abort flag).
static __device__ __noinline__ bool wait_global_at_least(const uint32_t* p, uint32_t target, Abort ab,
                                                         uint32_t site) {
  if (ld_acquire_gpu(p) >= target) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (ld_acquire_gpu(p) >= target) return true;
    if ((it & 15u) == 0u) {
      if (*ab.flag) return false;
      if (global_ns() - t0 > ab.limit_ns) {
        *ab.flag = 1u;
        if (ab.status) atomicCAS(ab.status, 0u, (site << 8) | kDevTimeout);
        return false;
      }
    }
    __nanosleep(32);
  }
}

}  // namespace lora
