// kernel_common.cuh — pieces shared by the decode kernels: bounded waits with
// a cluster-wide abort, remote shared-memory stores that complete on an
// mbarrier, 16-bit conversions, and the walk over a unit's segments.
#pragma once
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace mla {

constexpr uint64_t kTimeoutNs = 2000000000ull;  // a wait that runs this long aborts the step
constexpr uint64_t kDrainNs = 20000000ull;      // teardown waits after an abort

// One segment of a unit: tiles [t0, t1) of request b.
struct Seg {
  int b, t0, t1, n_tiles, slot;  // slot < 0: write the final output
};

// Walks the (request, tile-range) segments of one unit, in order.
struct SegIter {
  const int* req_meta;
  int B, b, begin_b, begin_t, end_b, end_t, first_split;
  __device__ SegIter(const DecodeParams& p, int unit) {
    const int* um = p.unit_meta + 5 * unit;
    req_meta = p.req_meta;
    B = p.batch;
    begin_b = um[0]; begin_t = um[1]; end_b = um[2]; end_t = um[3]; first_split = um[4];
    b = begin_b;
  }
  __device__ bool next(Seg& s) {
    while (b < B) {
      if (b > end_b || (b == end_b && end_t == 0)) return false;
      const int nt = req_meta[4 * b + 0];
      const int ns = req_meta[4 * b + 1];
      const int slot0 = req_meta[4 * b + 2];
      const int t0 = (b == begin_b) ? begin_t : 0;
      const int t1 = (b == end_b) ? end_t : nt;
      const int split = (b == begin_b) ? first_split : 0;
      s.b = b; s.t0 = t0; s.t1 = t1; s.n_tiles = nt;
      s.slot = (ns > 1) ? slot0 + split : -1;
      ++b;
      if (t0 < t1) return true;
    }
    return false;
  }
};

// Abort state of one CTA of a cluster.
struct Ctl {
  volatile uint32_t* abort;   // this CTA's abort flag (set by any CTA of the cluster)
  uint32_t abort_remote[3];   // the other CTAs' abort flags (cluster addresses)
  int n_remote;
  int* status;
};

__device__ __noinline__ inline void raise_timeout(const Ctl& c) {
  *c.abort = 1u;
  for (int i = 0; i < c.n_remote; ++i) st_cluster_u32(c.abort_remote[i], 1u);
  atomicCAS(c.status, 0, static_cast<int>(kStTimeout));
}

// Bounded wait: false if the wait ran out or the cluster is aborting.
template <bool kCluster>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& c) {
  if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 16; ++i)
      if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if (*c.abort) return false;
    if (globaltimer_ns() - t0 > kTimeoutNs) {
      raise_timeout(c);
      return false;
    }
  }
}

// Wait used only while tearing down after an abort: no abort check, short limit.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kDrainNs) return;
  }
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ANDs a flag over its threads.  Groups of warps that
// meet at named barriers after bounded waits vote with it, so that when one
// warp's wait fails they all leave at the same barrier (a warp that left
// alone would strand the others at their next bar.sync).
__device__ __forceinline__ bool named_bar_all(int id, int nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n"
      " bar.red.and.pred po, %2, %3, pi;\n selp.u32 %0, 1, 0, po;\n}"
      : "=r"(r) : "r"(v ? 1u : 0u), "r"(id), "r"(nthreads) : "memory");
  return r != 0;
}

template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Ctl& c) {
  return __all_sync(0xffffffffu, wait_bar<kCluster>(bar, parity, c));
}

// Remote shared-memory stores that complete on the destination CTA's mbarrier.
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
      ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d), "r"(bar) : "memory");
}
__device__ __forceinline__ void st_async_b32(uint32_t addr, uint32_t v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
               ::"r"(addr), "r"(v), "r"(bar) : "memory");
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// bf16x2 word -> fp16x2 word (exact for |v| in [2^-14, 65504]; smaller values
// become fp16 subnormals, absolute error <= 2^-25; larger ones overflow).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// acc + (both halves of a packed fp16x2 / bf16x2 word), each half widened
// exactly to fp32 by a mixed-precision add (one instruction per half)
__device__ __forceinline__ float add_f16x2_halves(float acc, uint32_t w) {
  asm("{\n .reg .f16 lo, hi;\n mov.b32 {lo, hi}, %1;\n add.rn.f32.f16 %0, lo, %0;\n add.rn.f32.f16 %0, hi, %0;\n}"
      : "+f"(acc) : "r"(w));
  return acc;
}
__device__ __forceinline__ float add_bf16x2_halves(float acc, uint32_t w) {
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n add.rn.f32.bf16 %0, lo, %0;\n add.rn.f32.bf16 %0, hi, %0;\n}"
      : "+f"(acc) : "r"(w));
  return acc;
}

__device__ __forceinline__ uint4 ld_shared_v4u(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
  return v;
}

}  // namespace mla
