// absorb_kernel.cu — the weight-absorption batched GEMMs on either side of
// absorbed-MLA decode ("DeepSeek V3/R1 Inference Efficiency (2)", §2.4.1,
// Compute: QKV projection Q''' = bmm(Q'', W_UK^T) and O projection
// O' = bmm(PV, W_UV)), and their C ABI (include/mla_absorb.h).
//
// Both are one small GEMM per head: M = the step's tokens (tiles of 128, the
// MMA's M), K and N from {128, 512}.  At decode batch sizes the weights
// (16 MiB each for 128 heads) dominate the bytes, so both kernels are bound
// by HBM and by latency: the design goal is every byte read once and loads
// in flight from the first cycle.  Operands arrive by TMA in the 128-byte
// swizzle the tensor cores read, products accumulate in TMEM (tcgen05.mma
// kind::f16, issued by one thread), and the epilogue goes TMEM -> registers
// -> bf16 -> swizzled shared memory -> TMA tensor store.
//
//   query side: persistent, one CTA per SM, work items of (token tile, head,
//     64 latent dims) in contiguous runs.  Warp 0 loads (A = q_nope tile
//     [128 tokens x 128 d], 32 KiB, once per (tile, head); B = W_UK[h] rows
//     [64 c x 128 d], K-major, 16 KiB per item) into rings of 2 and 8 slots
//     from right after the barrier set-up; warp 1 issues 8 MMAs of M128 N64 K16 per item into one of 8
//     TMEM accumulators; warps 2..5 drain accumulators (32 token rows each)
//     into per-warp staging and TMA stores; warp 6 copies the RoPE dims.
//   output side: CTA = (token tile, head), one per SM.  K = 512 latent dims
//     in 8 stages of 64 through a ring of 6 slots: A = O tile [128 tokens x
//     64 c] 16 KiB, B = W_UV[h] [64 c x 128 d] (MN-major: d contiguous)
//     16 KiB; 32 MMAs of M128 N128 K16.  Each O tile and weight is read once.
//
// Every wait is bounded: a wait that runs out records MLA_ERR_TIMEOUT in the
// caller's status word and the CTA tears down after short drain waits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "kernel_common.cuh"
#include "mla_absorb.h"

namespace mla {
namespace {

constexpr int kTokTile = 128;
constexpr int kDNope = 128;       // d
constexpr int kLatent = 512;      // c
constexpr int kRope = 64;
constexpr int kMaxAbsorbHeads = 128;
constexpr int kRowBytes = 128;    // one swizzle-atom row: 64 bf16
constexpr int kSlack = 1024;      // dynamic shared memory is re-aligned to 1024 B (128-byte swizzle atoms)

// ---- query side: persistent, one CTA per SM.  A work item is (token
// tile, head, 64 latent dims); items are numbered tile-major, then head, then
// latent slice, and each CTA takes a contiguous run of them, so the 8 items of
// one (tile, head) share the A tile it loaded.
constexpr int kQN = 64;                                 // latent dims per item (N of its MMAs)
constexpr int kQItemsPerHead = kLatent / kQN;           // 8
constexpr int kQASlot = 2 * kTokTile * kRowBytes;       // 32 KiB: 128 tokens x 128 d, two 64-d chunks
constexpr int kQBSlot = 2 * kQN * kRowBytes;            // 16 KiB: 64 latent rows x 128 d, two chunks
constexpr int kQASlots = 2, kQBSlots = 8, kQAcc = 8;    // 8 accumulators x 64 columns = all of TMEM
constexpr int kQStage = 32 * kRowBytes;                 // 4 KiB: one warp's 32 output rows of one item
constexpr int kQOffA = 0;
constexpr int kQOffB = kQOffA + kQASlots * kQASlot;     // 64 KiB
constexpr int kQOffStage = kQOffB + kQBSlots * kQBSlot; // 192 KiB, 4 warps x 2 buffers
constexpr int kQOffBar = kQOffStage + 4 * 2 * kQStage;  // 224 KiB
constexpr int kQNumBars = 2 * kQASlots + 2 * kQBSlots + 2 * kQAcc + 1;
constexpr int kQSmem = kQOffBar + kQNumBars * 8 + 16 + kSlack;
constexpr int kQThreads = 224;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue, warp 6 RoPE copy
constexpr uint32_t kQTmemCols = 512;
constexpr uint32_t kIdescQ = idesc_bf16(128, kQN, 0);
static_assert(kQSmem <= 232448, "shared memory");

// ---- output side: CTA = (token tile, head), all 128 output dims (N), the
// 512 latent dims (K) in 8 stages of 64 through a ring of 6 slots.
constexpr int kON = kDNope;                        // 128 output dims per CTA
constexpr int kOKStage = 64;                       // latent dims per stage (K)
constexpr int kOStages = kLatent / kOKStage;       // 8
constexpr int kOSlots = 6;
constexpr int kOAChunk = kTokTile * kRowBytes;     // 16 KiB: 128 tokens x 64 c
constexpr int kOBChunk = kOKStage * kRowBytes;     // 8 KiB: 64 c x 64 d
constexpr int kOSlotBytes = kOAChunk + 2 * kOBChunk;  // 32 KiB: A, then B as two 64-d chunks
constexpr int kOOffBar = kOSlots * kOSlotBytes;    // 192 KiB
constexpr int kOThreads = 128;
constexpr int kOSmem = kOOffBar + 128 + kSlack;
constexpr uint32_t kOTmemCols = 128;
constexpr uint32_t kIdescO = idesc_bf16(128, kON, 1);
static_assert(kOSmem <= 232448, "shared memory");

// 3-D tiled store from shared memory (completes in the thread's bulk group).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];"
               ::"l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(src)
               : "memory");
}

__device__ __forceinline__ void st_global_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
               ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// Epilogue of one 64-column slice: the warp's 32 TMEM lanes (token rows
// 32*warp .. +31), columns [col, col + 64), rounded to bf16 and written as
// row `row` of a 128-row, 128-byte-swizzled staging tile at `stage`.
__device__ __forceinline__ void stage_slice(uint32_t taddr, uint32_t stage, int row) {
  uint32_t lo[32], hi[32];
  tmem_ld32(taddr, lo);
  tmem_ld32(taddr + 32u, hi);
  tmem_wait_ld();
  const uint32_t rbase = stage + static_cast<uint32_t>(row) * kRowBytes;
  const uint32_t sw = static_cast<uint32_t>(row & 7);
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const uint32_t* s = u < 4 ? lo : hi;
    const int b = (u & 3) * 8;
    st_shared_v4(rbase + ((static_cast<uint32_t>(u) ^ sw) << 4),
                 pack_bf16x2(__uint_as_float(s[b + 0]), __uint_as_float(s[b + 1])),
                 pack_bf16x2(__uint_as_float(s[b + 2]), __uint_as_float(s[b + 3])),
                 pack_bf16x2(__uint_as_float(s[b + 4]), __uint_as_float(s[b + 5])),
                 pack_bf16x2(__uint_as_float(s[b + 6]), __uint_as_float(s[b + 7])));
  }
}

struct AbsorbParams {
  const uint16_t* q_pe;  // query side only (may be null)
  long long in_stride;   // q_pe row stride (elements)
  uint16_t* out;         // query side: destination of the RoPE copy
  long long out_stride;
  int num_tokens, num_heads;
  int* status;
};

// ============================================================ query side
__global__ void __launch_bounds__(kQThreads, 1)
mla_absorb_q_kernel(const __grid_constant__ AbsorbParams p, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_out) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t mis = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + mis;
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = p.num_heads;
  const long long n_items = static_cast<long long>((p.num_tokens + kTokTile - 1) / kTokTile) * H * kQItemsPerHead;
  const long long i0 = n_items * blockIdx.x / gridDim.x, i1 = n_items * (blockIdx.x + 1) / gridDim.x;

  const uint32_t bar0 = sbase + kQOffBar;
  auto a_full = [&](int s) { return bar0 + 8u * s; };
  auto a_empty = [&](int s) { return bar0 + 8u * (kQASlots + s); };
  auto b_full = [&](int s) { return bar0 + 8u * (2 * kQASlots + s); };
  auto b_empty = [&](int s) { return bar0 + 8u * (2 * kQASlots + kQBSlots + s); };
  auto acc_full = [&](int s) { return bar0 + 8u * (2 * kQASlots + 2 * kQBSlots + s); };
  auto acc_empty = [&](int s) { return bar0 + 8u * (2 * kQASlots + 2 * kQBSlots + kQAcc + s); };
  const uint32_t bar_drain = bar0 + 8u * (kQNumBars - 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kQOffBar + kQNumBars * 8);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kQOffBar + kQNumBars * 8 + 4);
  auto a_slot = [&](int s) { return sbase + static_cast<uint32_t>(kQOffA + s * kQASlot); };
  auto b_slot = [&](int s) { return sbase + static_cast<uint32_t>(kQOffB + s * kQBSlot); };

  Ctl ctl;
  ctl.abort = abort_flag;
  ctl.n_remote = 0;
  ctl.status = p.status;

  // TMA producer state: item pi is the next to load, pk its index in this
  // CTA's run, pa the number of A tiles loaded, p_prev the (tile, head) of the last one
  long long pi = i0, p_prev = -1;
  int pk = 0, pa = 0;
  auto load_b = [&](long long i, int k) {
    const int s = k % kQBSlots;
    const int c8 = static_cast<int>(i % kQItemsPerHead);
    const int h = static_cast<int>((i / kQItemsPerHead) % H);
    const int row = h * kLatent + c8 * kQN;
    mbar_arrive_expect_tx(b_full(s), kQBSlot);
    tma_load_2d(b_slot(s), &tm_w, 0, row, b_full(s));
    tma_load_2d(b_slot(s) + kQBSlot / 2, &tm_w, 64, row, b_full(s));
  };
  // The weight slices of the first kQBSlots items go out before the wait for
  // the previous kernel (programmatic dependent launch; the weights are not
  // written by it); then the loads follow in item order, each once its slot
  // is free.  False if a wait ran out.
  auto produce = [&]() -> bool {
    for (int k = 0; k < kQBSlots && i0 + k < i1; ++k) load_b(i0 + k, k);
    grid_dependency_wait();
    for (; pi < i1; ++pi, ++pk) {
      const long long th = pi / kQItemsPerHead;  // tile * H + head
      if (th != p_prev) {
        if (pa >= kQASlots) {
          if (!wait_bar<false>(a_empty(pa % kQASlots), ((pa / kQASlots) - 1) & 1, ctl)) return false;
        }
        const int s = pa % kQASlots;
        const int h = static_cast<int>(th % H), t0 = static_cast<int>(th / H) * kTokTile;
        mbar_arrive_expect_tx(a_full(s), kQASlot);
        tma_load_3d(a_slot(s), &tm_q, 0, h, t0, a_full(s));
        tma_load_3d(a_slot(s) + kQASlot / 2, &tm_q, 64, h, t0, a_full(s));
        ++pa;
        p_prev = th;
      }
      if (pk >= kQBSlots) {
        if (!wait_bar<false>(b_empty(pk % kQBSlots), ((pk / kQBSlots) - 1) & 1, ctl)) return false;
        load_b(pi, pk);
      }
    }
    return true;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kQNumBars; ++i) {
      const bool acc_e = bar0 + 8u * i >= acc_empty(0) && bar0 + 8u * i < acc_empty(kQAcc);
      mbar_init(bar0 + 8u * i, acc_e ? 4 : 1);  // accumulators are released by each epilogue warp
    }
    *abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  // The producer starts loading at once; TMEM is allocated meanwhile and its
  // address reaches the MMA and epilogue warps (1..5) through named barrier 1.
  uint32_t tmem = 0;
  if (warp >= 1 && warp <= 5) {
    if (warp == 1) {
      tmem_alloc(smem_u32(tmem_slot), kQTmemCols);
      tmem_relinquish();
    }
    tc_fence_before();
    named_bar_sync(1, 5 * 32);
    tc_fence_after();
    tmem = *tmem_slot;
  }

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_w);
      tma_prefetch_desc(&tm_out);
      produce();
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      long long prev = -1;
      int na = 0, k = 0;
      for (long long i = i0; i < i1; ++i, ++k) {
        const long long th = i / kQItemsPerHead;
        if (th != prev) {
          if (na > 0) umma_commit(a_empty((na - 1) % kQASlots));  // the previous A tile is done with
          if (!wait_bar<false>(a_full(na % kQASlots), (na / kQASlots) & 1, ctl)) break;
          ++na;
          prev = th;
        }
        const int bs = k % kQBSlots, acc = k % kQAcc;
        if (!wait_bar<false>(b_full(bs), (k / kQBSlots) & 1, ctl)) break;
        if (k >= kQAcc && !wait_bar<false>(acc_empty(acc), ((k / kQAcc) - 1) & 1, ctl)) break;
        tc_fence_after();
        const uint64_t ad = smem_desc(a_slot((na - 1) % kQASlots), 16u, 1024u);
        const uint64_t bd = smem_desc(b_slot(bs), 16u, 1024u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_f16(tmem + static_cast<uint32_t>(acc * kQN),
                   ad + static_cast<uint64_t>(((kk >> 2) * (kQASlot / 2) + (kk & 3) * 32) >> 4),
                   bd + static_cast<uint64_t>(((kk >> 2) * (kQBSlot / 2) + (kk & 3) * 32) >> 4), kIdescQ,
                   kk != 0 ? 1u : 0u);
        umma_commit(b_empty(bs));
        umma_commit(acc_full(acc));
      }
      umma_commit(bar_drain);  // arrives once every MMA issued above has completed
    }
    __syncwarp();
  } else if (warp < 6) {
    // epilogue: warp w reads TMEM lanes 32 * (w % 4) .. +31 = those token rows
    const int q = warp & 3;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    int k = 0;
    for (long long i = i0; i < i1; ++i, ++k) {
      const int c8 = static_cast<int>(i % kQItemsPerHead);
      const long long th = i / kQItemsPerHead;
      const int h = static_cast<int>(th % H), t0 = static_cast<int>(th / H) * kTokTile;
      const int acc = k % kQAcc;
      if (!warp_wait(acc_full(acc), (k / kQAcc) & 1, ctl)) break;
      tc_fence_after();
      uint32_t lo[32], hi[32];
      tmem_ld32(tl + static_cast<uint32_t>(acc * kQN), lo);
      tmem_ld32(tl + static_cast<uint32_t>(acc * kQN + 32), hi);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(acc_empty(acc));  // the accumulator may take the item after next
        bulk_wait_read_1();           // this staging buffer's previous store has read it
      }
      __syncwarp();
      const uint32_t stg = sbase + static_cast<uint32_t>(kQOffStage + (q * 2 + (k & 1)) * kQStage);
      const uint32_t rbase = stg + static_cast<uint32_t>(lane) * kRowBytes;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t* src = u < 4 ? lo : hi;
        const int b = (u & 3) * 8;
        st_shared_v4(rbase + ((static_cast<uint32_t>(u) ^ static_cast<uint32_t>(lane & 7)) << 4),
                     pack_bf16x2(__uint_as_float(src[b + 0]), __uint_as_float(src[b + 1])),
                     pack_bf16x2(__uint_as_float(src[b + 2]), __uint_as_float(src[b + 3])),
                     pack_bf16x2(__uint_as_float(src[b + 4]), __uint_as_float(src[b + 5])),
                     pack_bf16x2(__uint_as_float(src[b + 6]), __uint_as_float(src[b + 7])));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (t0 + q * 32 < p.num_tokens) tma_store_3d(&tm_out, stg, c8 * kQN, h, t0 + q * 32);
        bulk_commit();
      }
    }
    if (lane == 0) bulk_wait_read();  // staging stays valid until the stores have read it
    __syncwarp();

  } else if (p.q_pe != nullptr) {
    // RoPE dims pass through unchanged, once per (tile, head): one 128-byte row per lane at a time
    grid_dependency_wait();
    for (long long i = i0; i < i1; ++i) {
      if (i % kQItemsPerHead != 0) continue;
      const long long th = i / kQItemsPerHead;
      const int h = static_cast<int>(th % H), t0 = static_cast<int>(th / H) * kTokTile;
      for (int r = lane; r < kTokTile; r += 32) {
        const int t = t0 + r;
        if (t >= p.num_tokens) break;
        const long long row = static_cast<long long>(t) * H + h;
        const uint16_t* src = p.q_pe + row * p.in_stride;
        uint16_t* dst = p.out + row * p.out_stride + kLatent;
        uint4 v[kRope / 8];
#pragma unroll
        for (int j = 0; j < kRope / 8; ++j) v[j] = ld_global_nc_v4(src + 8 * j);
#pragma unroll
        for (int j = 0; j < kRope / 8; ++j) st_global_v4(dst + 8 * j, v[j]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 32) drain_bar(bar_drain, 0u);  // MMAs finish before TMEM is released
  if (threadIdx.x == 0 && *abort_flag) {
    // teardown after a wait ran out: loads still in flight land before the CTA exits
    const int nb = pk > kQBSlots ? pk : static_cast<int>(i1 - i0 < kQBSlots ? i1 - i0 : kQBSlots);
    for (int s = 0; s < kQBSlots && s < nb; ++s) drain_bar(b_full(s), (((nb - 1 - s) / kQBSlots)) & 1);
    for (int s = 0; s < kQASlots && s < pa; ++s) drain_bar(a_full(s), (((pa - 1 - s) / kQASlots)) & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kQTmemCols);
  }
}

// ============================================================ output side
__global__ void __launch_bounds__(kOThreads, 1)
mla_absorb_o_kernel(const __grid_constant__ AbsorbParams p, const __grid_constant__ CUtensorMap tm_o,
                    const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_out) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t mis = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + mis;
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kTokTile, h = blockIdx.y;
  const uint32_t bar_full = sbase + kOOffBar;          // kOSlots
  const uint32_t bar_empty = bar_full + 8 * kOSlots;   // kOSlots
  const uint32_t bar_mma = bar_empty + 8 * kOSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOOffBar + 16 * kOSlots + 8);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kOOffBar + 16 * kOSlots + 12);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kOSlots; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, 1);
    }
    mbar_init(bar_mma, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  Ctl ctl;
  ctl.abort = abort_flag;
  ctl.n_remote = 0;
  ctl.status = p.status;
  auto slot_a = [&](int s) { return sbase + static_cast<uint32_t>(s * kOSlotBytes); };
  auto slot_b = [&](int s) { return sbase + static_cast<uint32_t>(s * kOSlotBytes + kOAChunk); };

  // the producer starts loading at once; TMEM reaches warps 1..3 through named barrier 1
  int issued = 0;  // stages whose activation tile was requested
  uint32_t tmem = 0;
  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      tma_prefetch_desc(&tm_o);
      tma_prefetch_desc(&tm_w);
      tma_prefetch_desc(&tm_out);
      auto load_w = [&](int s) {
        const uint32_t bar = bar_full + 8 * (s % kOSlots);
        const int row = h * kLatent + kOKStage * s;
        mbar_arrive_expect_tx(bar, kOSlotBytes);  // the stage's weight and activation bytes
        tma_load_2d(slot_b(s % kOSlots), &tm_w, 0, row, bar);
        tma_load_2d(slot_b(s % kOSlots) + kOBChunk, &tm_w, 64, row, bar);
      };
      // weights of the first stages before the wait for the previous kernel
      // (programmatic dependent launch; it does not write the weights)
      for (int s = 0; s < kOSlots && s < kOStages; ++s) load_w(s);
      grid_dependency_wait();
      for (int s = 0; s < kOStages; ++s) {
        const int slot = s % kOSlots;
        if (s >= kOSlots) {
          if (!wait_bar<false>(bar_empty + 8 * slot, ((s / kOSlots) - 1) & 1, ctl)) break;
          load_w(s);
        }
        tma_load_3d(slot_a(slot), &tm_o, kOKStage * s, h, t0, bar_full + 8 * slot);
        issued = s + 1;
      }
    }
    __syncwarp();
  } else {
    if (warp == 1) {
      tmem_alloc(smem_u32(tmem_slot), kOTmemCols);
      tmem_relinquish();
    }
    tc_fence_before();
    named_bar_sync(1, 3 * 32);
    tc_fence_after();
    tmem = *tmem_slot;
    if (warp == 1) {
      if (lane == 0) {  // MMA issuer
        for (int s = 0; s < kOStages; ++s) {
          const int slot = s % kOSlots;
          if (!wait_bar<false>(bar_full + 8 * slot, (s / kOSlots) & 1, ctl)) break;
          tc_fence_after();
          const uint64_t ad = smem_desc(slot_a(slot), 16u, 1024u);
          const uint64_t bd = smem_desc(slot_b(slot), static_cast<uint32_t>(kOBChunk), 1024u);  // MN-major
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_f16(tmem, ad + static_cast<uint64_t>((32 * kk) >> 4), bd + static_cast<uint64_t>((2048 * kk) >> 4),
                     kIdescO, (s | kk) != 0 ? 1u : 0u);
          umma_commit(bar_empty + 8 * slot);
        }
        umma_commit(bar_mma);  // arrives once every MMA issued above has completed
      }
      __syncwarp();
    }
  }
  // all four warps drain the accumulator (TMEM lanes 32 * warp .. +31)
  tc_fence_before();
  named_bar_sync(2, kOThreads);
  tc_fence_after();
  tmem = *tmem_slot;

  // epilogue: two 64-column slices staged in slot 0 (free once every MMA has completed)
  bool ok = warp_wait(bar_mma, 0u, ctl) && *abort_flag == 0u;
  tc_fence_after();
  const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  if (ok) {
    stage_slice(tl, slot_a(0), warp * 32 + lane);
    stage_slice(tl + 64u, slot_a(0) + kOAChunk, warp * 32 + lane);
    fence_proxy_async_smem();
  }
  ok = named_bar_all(3, kOThreads, ok);
  if (threadIdx.x == 0) {
    if (ok) {
      tma_store_3d(&tm_out, slot_a(0), 0, h, t0);
      tma_store_3d(&tm_out, slot_a(0) + kOAChunk, 64, h, t0);
      bulk_commit();
      bulk_wait_read();
    } else {
      // teardown after a wait ran out: loads still in flight land before the CTA exits
      for (int s = issued > kOSlots ? issued - kOSlots : 0; s < issued; ++s)
        drain_bar(bar_full + 8 * (s % kOSlots), (s / kOSlots) & 1);
      drain_bar(bar_mma, 0u);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kOTmemCols);
  }
}

// ============================================================ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

constexpr int kMaxDev = 64;
struct AbsorbDevice {
  std::once_flag once;
  int status = MLA_OK;
  int sms = 0;
};
AbsorbDevice g_abs_dev[kMaxDev];

// Compute capability 10.3 check and kernel attributes, once per device.
int absorb_device_ready() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return MLA_ERR_DEVICE;
  AbsorbDevice& st = g_abs_dev[dev];
  std::call_once(st.once, [&st, dev] {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        major != 10 || minor != 3) {
      st.status = MLA_ERR_DEVICE;
      return;
    }
    if (cudaFuncSetAttribute(mla_absorb_q_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(mla_absorb_o_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kOSmem) !=
            cudaSuccess) {
      cudaGetLastError();
      st.status = MLA_ERR_CUDA;
      return;
    }
    if (cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || st.sms < 1)
      st.status = MLA_ERR_DEVICE;
  });
  return st.status;
}

int absorb_sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  return g_abs_dev[dev].sms;
}

// A token-major activation [T, H, dims] with rows `stride` elements apart,
// as 3-D boxes of {64 dims, 1 head, box_tokens tokens} in the 128-byte swizzle.
int encode_act(CUtensorMap* m, const void* base, uint64_t dims, int64_t stride, int heads, int tokens,
               uint32_t box_tokens) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return MLA_ERR_CUDA;
  const cuuint64_t size[3] = {dims, static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(tokens)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(stride) * 2,
                                 static_cast<cuuint64_t>(stride) * 2 * static_cast<cuuint64_t>(heads)};
  const cuuint32_t box[3] = {64u, 1u, box_tokens};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), size, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_CUDA;
}

// A weight [H, 512, 128] as 2-D [H * 512 rows, 128 columns], boxes of
// {64 columns, box_rows rows} in the 128-byte swizzle.
int encode_weight(CUtensorMap* m, const void* base, int heads, uint32_t box_rows) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return MLA_ERR_CUDA;
  const cuuint64_t size[2] = {static_cast<cuuint64_t>(kDNope), static_cast<cuuint64_t>(heads) * kLatent};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDNope) * 2};
  const cuuint32_t box[2] = {64u, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), size, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_CUDA;
}

// Launch as a programmatic dependent of the kernel before it on the stream:
// the kernel's set-up and weight loads overlap that kernel's tail, and it
// waits for that kernel (griddepcontrol.wait) before touching activations.
int launch_dependent(void (*kernel)(AbsorbParams, CUtensorMap, CUtensorMap, CUtensorMap), dim3 grid, dim3 block,
                     int smem, mla_stream_t stream, const AbsorbParams& p, const CUtensorMap& a,
                     const CUtensorMap& b, const CUtensorMap& c) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, p, a, b, c) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool stride_ok(int64_t s, int64_t min) { return s >= min && (s & 7) == 0 && s <= (int64_t{1} << 30); }

int common_checks(int num_tokens, int num_heads, const int* status) {
  if (num_tokens < 0 || !status || (reinterpret_cast<uintptr_t>(status) & 3u) != 0) return MLA_ERR_INVALID_ARG;
  if (num_heads < 1 || num_heads > kMaxAbsorbHeads) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

int mla_absorb_q(const void* q_nope, const void* q_pe, int64_t q_stride, const void* w_uk, int num_tokens,
                 int num_heads, void* out, int64_t out_stride, int* status, mla_stream_t stream) {
  int rc = common_checks(num_tokens, num_heads, status);
  if (rc != MLA_OK) return rc;
  if (!q_nope || !w_uk || !out || !al16(q_nope) || !al16(w_uk) || !al16(out) || (q_pe && !al16(q_pe)))
    return MLA_ERR_INVALID_ARG;
  if (!stride_ok(q_stride, kDNope) || !stride_ok(out_stride, q_pe ? kLatent + kRope : kLatent))
    return MLA_ERR_INVALID_ARG;
  if ((rc = absorb_device_ready()) != MLA_OK) return rc;
  if (num_tokens == 0) return MLA_OK;
  CUtensorMap tm_q, tm_w, tm_out;
  if ((rc = encode_act(&tm_q, q_nope, kDNope, q_stride, num_heads, num_tokens, kTokTile)) != MLA_OK ||
      (rc = encode_weight(&tm_w, w_uk, num_heads, kQN)) != MLA_OK ||
      (rc = encode_act(&tm_out, out, kLatent, out_stride, num_heads, num_tokens, 32)) != MLA_OK)
    return rc;
  AbsorbParams p;
  p.q_pe = static_cast<const uint16_t*>(q_pe);
  p.in_stride = q_stride;
  p.out = static_cast<uint16_t*>(out);
  p.out_stride = out_stride;
  p.num_tokens = num_tokens;
  p.num_heads = num_heads;
  p.status = status;
  // one CTA per SM (its shared memory admits no second), each a contiguous run of items
  const long long items = static_cast<long long>((num_tokens + kTokTile - 1) / kTokTile) * num_heads * kQItemsPerHead;
  const int grid = static_cast<int>(items < absorb_sm_count() ? items : absorb_sm_count());
  return launch_dependent(mla_absorb_q_kernel, dim3(grid), dim3(kQThreads), kQSmem, stream, p, tm_q, tm_w, tm_out);
}

int mla_absorb_o(const void* o, int64_t o_stride, const void* w_uv, int num_tokens, int num_heads, void* out,
                 int64_t out_stride, int* status, mla_stream_t stream) {
  int rc = common_checks(num_tokens, num_heads, status);
  if (rc != MLA_OK) return rc;
  if (!o || !w_uv || !out || !al16(o) || !al16(w_uv) || !al16(out)) return MLA_ERR_INVALID_ARG;
  if (!stride_ok(o_stride, kLatent) || !stride_ok(out_stride, kDNope)) return MLA_ERR_INVALID_ARG;
  if ((rc = absorb_device_ready()) != MLA_OK) return rc;
  if (num_tokens == 0) return MLA_OK;
  CUtensorMap tm_o, tm_w, tm_out;
  if ((rc = encode_act(&tm_o, o, kLatent, o_stride, num_heads, num_tokens, kTokTile)) != MLA_OK ||
      (rc = encode_weight(&tm_w, w_uv, num_heads, kOKStage)) != MLA_OK ||
      (rc = encode_act(&tm_out, out, kDNope, out_stride, num_heads, num_tokens, kTokTile)) != MLA_OK)
    return rc;
  AbsorbParams p = {};
  p.num_tokens = num_tokens;
  p.num_heads = num_heads;
  p.status = status;
  const dim3 grid((num_tokens + kTokTile - 1) / kTokTile, num_heads, 1);
  return launch_dependent(mla_absorb_o_kernel, grid, dim3(kOThreads), kOSmem, stream, p, tm_o, tm_w, tm_out);
}

}  // extern "C"
