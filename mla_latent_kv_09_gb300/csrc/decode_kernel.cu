// decode_kernel.cu — weight-absorbed MLA decode attention on sm_103a.
//
// What it computes ("DeepSeek V3/R1 Inference Efficiency (2)", §2.4.1,
// Compute, "MLA/MQA attention"): every request's 128 query heads (576 dims:
// 512 latent + 64 RoPE) attend over the request's cached latent rows; scores
// contract all 576 dims, values are the first 512 dims of the same row.
// Cached rows sit in 64-token pages reached through a block table.
//
// How (one work unit = one 2-CTA cluster on a pair of SMs):
//   * O = 128 heads x 512 fp32 fills a whole SM's tensor memory, so the pair
//     splits the row: CTA 0 owns latent dims [0, 256) and O columns [0, 256),
//     CTA 1 owns dims [256, 576) (latent 256..511 + RoPE) and O columns
//     [256, 512).  Each cache byte is fetched from HBM exactly once.
//   * Per 64-token tile: each CTA computes its partial scores
//     S_r = Q[:, dims_r] K[:, dims_r]^T on tcgen05 (M=128, N=64, K=256/320,
//     fp32 in TMEM), the two partials are swapped through distributed shared
//     memory and added (fp32 addition commutes, so both CTAs hold bit-equal
//     scores and take identical softmax decisions), the online softmax runs
//     in fp32 (exp2 domain, running max with a lazy-rescale threshold), P goes
//     to shared memory as bf16 and each CTA accumulates O_r += P V_r on
//     tcgen05 (M=128, N=256, K=64) with V_r read from the same smem tile.
//   * A persistent grid: each unit walks a contiguous range of (request,
//     tile) work from the plan; a request cut by a range boundary writes a
//     normalised fp32 partial plus its LSE, merged later by the combine
//     kernel (the split-K remedy of "The 31-Millisecond Smoking Gun").
//
// Warp roles (288 threads): warps 0-3 softmax / epilogue (thread i owns head
// row i = TMEM lane i), warp 4 issues MMAs and owns TMEM, warps 5-8 load
// (dense: one thread drives TMA; sparse: 128 threads gather rows).
#include <cuda_runtime.h>

#include "common.cuh"
#include "plan.cuh"
#include "ptx.cuh"

namespace mla {

constexpr int kQChunkBytes = kHeads * 128;   // 128 rows x 64 bf16
constexpr int kKvChunkBytes = kPage * 128;   // 64 rows x 64 bf16
constexpr int kNqMax = 5;
constexpr int kStages = 2;
constexpr int kQBytes = kNqMax * kQChunkBytes;       // 81920
constexpr int kStageBytes = kNqMax * kKvChunkBytes;  // 40960
constexpr int kPBytes = kHeads * 128;                // 128 rows x 64 bf16
constexpr int kXBytes = kHeads * 64 * 4;             // 128 rows x 64 fp32

constexpr int kOffQ = 0;
constexpr int kOffKv = kOffQ + kQBytes;
constexpr int kOffP = kOffKv + kStages * kStageBytes;
constexpr int kOffX = kOffP + 2 * kPBytes;
constexpr int kOffBar = kOffX + kXBytes;
constexpr int kBarBytes = 256;
constexpr int kOffMask = kOffBar + kBarBytes;  // sparse: 64-bit row-valid mask per stage
constexpr int kMaskBytes = 16;
constexpr int kSmemBytes = kOffMask + kMaskBytes + 1024;  // + alignment slack

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;
constexpr uint32_t kColS = 256;  // two 64-column score buffers

constexpr int kNumThreads = 288;
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the max grows by > 2^8
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr uint64_t kDrainNs = 20000000ull;

enum Bar {
  kKvFull0, kKvFull1, kKvEmpty0, kKvEmpty1, kQFull, kQEmpty, kSFull0, kSFull1, kSFree0,
  kSFree1, kPFull0, kPFull1, kPFree0, kPFree1, kOFull, kOFree, kXFull, kXFree, kMmaDone,
  kNumBars
};
static_assert(kNumBars * 8 + 16 <= kBarBytes, "barrier area");

constexpr uint32_t kIdescQK = idesc_bf16(128, 64, 0);
constexpr uint32_t kIdescPV = idesc_bf16(128, 256, 1);

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

struct Ctl {
  volatile uint32_t* abort;  // this CTA's abort flag (set by either CTA)
  uint32_t abort_remote;     // the peer's abort flag (cluster address)
  int* status;
};

__device__ __noinline__ void raise_timeout(const Ctl& c) {
  *c.abort = 1u;
  st_cluster_u32(c.abort_remote, 1u);
  atomicCAS(c.status, 0, static_cast<int>(kStTimeout));
}

// Bounded wait: false if the wait ran out or the CTA pair is aborting.
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

template <bool kSparse>
__global__ void __launch_bounds__(kNumThreads, 1)
mla_decode_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_kv) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int U = p.num_units;
  const int cluster_id = blockIdx.x >> 1;
  const int unit = cluster_id % U;
  const int tok = cluster_id / U;
  const int nq = rank == 0 ? 4 : 5;          // 64-dim chunks this CTA owns
  const int chunk0 = rank == 0 ? 0 : 4;

  {  // a unit with no work leaves at once (both CTAs see the same range)
    const int* um = p.unit_meta + 5 * unit;
    if (um[0] >= p.batch || (um[0] == um[2] && um[1] >= um[3])) return;
  }

  const uint32_t sQ = sbase + kOffQ;
  const uint32_t sKv = sbase + kOffKv;
  const uint32_t sP = sbase + kOffP;
  const uint32_t sX = sbase + kOffX;
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * static_cast<uint32_t>(i); };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * kNumBars);
  // misc[0] = TMEM base address, misc[1] = abort flag

  if (threadIdx.x == 0) {
    mbar_init(bar(kKvFull0), kSparse ? 128 : 1);
    mbar_init(bar(kKvFull1), kSparse ? 128 : 1);
    mbar_init(bar(kKvEmpty0), 1);
    mbar_init(bar(kKvEmpty1), 1);
    mbar_init(bar(kQFull), 1);
    mbar_init(bar(kQEmpty), 1);
    mbar_init(bar(kSFull0), 1);
    mbar_init(bar(kSFull1), 1);
    mbar_init(bar(kSFree0), 128);
    mbar_init(bar(kSFree1), 128);
    mbar_init(bar(kPFull0), 128);
    mbar_init(bar(kPFull1), 128);
    mbar_init(bar(kPFree0), 1);
    mbar_init(bar(kPFree1), 1);
    mbar_init(bar(kOFull), 1);
    mbar_init(bar(kOFree), 128);
    mbar_init(bar(kXFull), 128);
    mbar_init(bar(kXFree), 128);
    mbar_init(bar(kMmaDone), 1);
    misc[1] = 0u;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(&misc[0]), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 5 && lane == 0 && !kSparse) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kv);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = misc[0];

  Ctl ctl;
  ctl.abort = &misc[1];
  ctl.abort_remote = mapa(smem_u32(&misc[1]), peer);
  ctl.status = p.ws_hdr + kHdrStatus;

  if (warp < 4) {
    // ===================================================== softmax / epilogue
    const int row = threadIdx.x;  // head = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t x_row = sX + static_cast<uint32_t>(row) * 256u;
    const uint32_t x_row_remote = mapa(x_row, peer);
    const uint32_t xfull_remote = mapa(bar(kXFull), peer);
    const uint32_t xfree_remote = mapa(bar(kXFree), peer);
    const float NEG_INF = -__int_as_float(0x7f800000);
    SegIter it(p, unit);
    Seg sg;
    uint32_t g = 0, nseg = 0;
    bool ok = true;
    while (ok && it.next(sg)) {
      const int L = max(p.cache_lens[sg.b], 0);
      const int vis = p.causal ? L - p.s_q + tok + 1 : L;
      // z: sum of the bf16-rounded weights (normalises O, whose PV product uses
      // exactly those weights); zx: sum of the unrounded weights (for the LSE)
      float m_used = NEG_INF, z = 0.f, zx = 0.f;
      for (int j = sg.t0; j < sg.t1; ++j, ++g) {
        const uint32_t sb = g & 1u, ph = (g >> 1) & 1u;
        ok = __all_sync(0xffffffffu, wait_bar<false>(bar(kSFull0 + sb), ph, ctl));
        if (kSparse && ok) ok = __all_sync(0xffffffffu, wait_bar<false>(bar(kKvFull0 + sb), ph, ctl));
        if (!ok) break;
        tc_fence_after();
        float s[64];
        {
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + kColS + 64u * sb, r);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) s[c] = __uint_as_float(r[c]);
          tmem_ld32(tmem + lane_base + kColS + 64u * sb + 32u, r);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) s[32 + c] = __uint_as_float(r[c]);
        }
        tc_fence_before();
        mbar_arrive(bar(kSFree0 + sb));

        // ---- swap partial scores with the peer CTA through DSMEM
        if (!(ok = __all_sync(0xffffffffu, wait_bar<true>(bar(kXFree), (g & 1u) ^ 1u, ctl)))) break;
#pragma unroll
        for (int c = 0; c < 16; ++c)
          st_cluster_v4(x_row_remote + ((static_cast<uint32_t>(c) ^ (row & 15)) << 4), s[4 * c],
                        s[4 * c + 1], s[4 * c + 2], s[4 * c + 3]);
        mbar_arrive_remote(xfull_remote);
        if (!(ok = __all_sync(0xffffffffu, wait_bar<true>(bar(kXFull), g & 1u, ctl)))) break;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float4 v = ld_shared_v4f(x_row + ((static_cast<uint32_t>(c) ^ (row & 15)) << 4));
          s[4 * c] += v.x; s[4 * c + 1] += v.y; s[4 * c + 2] += v.z; s[4 * c + 3] += v.w;
        }
        mbar_arrive_remote(xfree_remote);

        // ---- mask, scale to the exp2 domain, running max
        float mt = NEG_INF;
        if (kSparse) {
          // rows the loaders actually fetched (index in [0, len), page in the pool)
          const unsigned long long vmask =
              *reinterpret_cast<const volatile unsigned long long*>(smem + kOffMask + 8 * sb);
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const float t = ((vmask >> c) & 1ull) ? s[c] * p.scale_log2 : NEG_INF;
            s[c] = t;
            mt = fmaxf(mt, t);
          }
        } else {
          const int nvalid = vis - j * 64;
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const float t = c < nvalid ? s[c] * p.scale_log2 : NEG_INF;
            s[c] = t;
            mt = fmaxf(mt, t);
          }
        }

        // ---- online softmax with a lazy rescale: the reference max m_used
        // moves only when a score exceeds it by more than 2^8, so P <= 256.
        bool resc = false;
        float alpha = 1.f;
        if (mt > m_used + kRescaleLog2 || (m_used == NEG_INF && mt != NEG_INF)) {
          alpha = (m_used == NEG_INF) ? 0.f : ex2_approx(m_used - mt);
          resc = (m_used != NEG_INF) && (j != sg.t0);
          m_used = mt;
          z *= alpha;
          zx *= alpha;
        }
        uint32_t pk[32];
        if (m_used == NEG_INF) {
#pragma unroll
          for (int c = 0; c < 32; ++c) pk[c] = 0u;
        } else {
          float zs = 0.f, ze = 0.f;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float p0 = ex2_approx(s[2 * c] - m_used);
            const float p1 = ex2_approx(s[2 * c + 1] - m_used);
            pk[c] = pack_bf16x2(p0, p1);
            zs += __uint_as_float(pk[c] << 16) + __uint_as_float(pk[c] & 0xffff0000u);
            ze += p0 + p1;
          }
          z += zs;
          zx += ze;
        }

        // ---- rescale O (warp-uniform: tcgen05.ld/st are warp-collective)
        if (__any_sync(0xffffffffu, resc)) {
          const uint32_t gp = g - 1u;
          if (!(ok = __all_sync(0xffffffffu,
                                wait_bar<false>(bar(kPFree0 + (gp & 1u)), (gp >> 1) & 1u, ctl))))
            break;
          tc_fence_after();
          const float a = resc ? alpha : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t r[32];
            const uint32_t ta = tmem + lane_base + kColO + 32u * cc;
            tmem_ld32(ta, r);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * a);
            tmem_st32(ta, r);
          }
          tmem_wait_st();
        }

        // ---- P -> shared memory (K-major, 128-byte swizzle), after PV(g-2)
        if (!(ok = __all_sync(0xffffffffu, wait_bar<false>(bar(kPFree0 + sb), ph ^ 1u, ctl)))) break;
        {
          const uint32_t prow = sP + sb * kPBytes + static_cast<uint32_t>(row) * 128u;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            st_shared_v4(prow + ((static_cast<uint32_t>(k) ^ (row & 7)) << 4), pk[4 * k],
                         pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        }
        // rows past the end of the cache in the request's last page may hold
        // anything (even NaN); zero their value part so 0 * V stays 0
        if (!kSparse && j == sg.n_tiles - 1 && L < (j + 1) * 64) {
          const int r0 = L - j * 64;
          const int n = (64 - r0) * 32;
          const uint32_t st = sKv + sb * kStageBytes;
          for (int e = row; e < n; e += 128) {
            const int rr = r0 + (e >> 5), c16 = e & 31;
            st_shared_zero16(st + (c16 >> 3) * kKvChunkBytes + rr * 128 +
                             (((c16 & 7) ^ (rr & 7)) << 4));
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(kPFull0 + sb));

        // ---- segment epilogue
        if (j == sg.t1 - 1) {
          if (!(ok = __all_sync(0xffffffffu, wait_bar<false>(bar(kOFull), nseg & 1u, ctl)))) break;
          tc_fence_after();
          const float inv = z > 0.f ? 1.f / z : 0.f;
          const float lse = zx > 0.f ? (m_used + log2f(zx)) * 0.69314718055994531f : NEG_INF;
          const long long bt_row = static_cast<long long>(sg.b) * p.s_q + tok;
          if (sg.slot < 0) {
            const long long o_off = (bt_row * kHeads + row) * kDv + rank * kVcolsPerCta;
#pragma unroll 1
            for (int cc = 0; cc < 8; ++cc) {
              uint32_t r[32];
              tmem_ld32(tmem + lane_base + kColO + 32u * cc, r);
              tmem_wait_ld();
              if (p.out_fp32) {
                float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + o_off + 32 * cc);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                  dst[k] = make_float4(__uint_as_float(r[4 * k]) * inv, __uint_as_float(r[4 * k + 1]) * inv,
                                       __uint_as_float(r[4 * k + 2]) * inv, __uint_as_float(r[4 * k + 3]) * inv);
              } else {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + o_off + 32 * cc);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  dst[k] = make_uint4(
                      pack_bf16x2(__uint_as_float(r[8 * k + 0]) * inv, __uint_as_float(r[8 * k + 1]) * inv),
                      pack_bf16x2(__uint_as_float(r[8 * k + 2]) * inv, __uint_as_float(r[8 * k + 3]) * inv),
                      pack_bf16x2(__uint_as_float(r[8 * k + 4]) * inv, __uint_as_float(r[8 * k + 5]) * inv),
                      pack_bf16x2(__uint_as_float(r[8 * k + 6]) * inv, __uint_as_float(r[8 * k + 7]) * inv));
              }
            }
            if (rank == 0) p.lse[bt_row * kHeads + row] = lse;
          } else if (sg.slot < 2 * U) {  // the plan never uses more than 2 * (U - 1) slots
            const long long prow_id = static_cast<long long>(sg.slot) * p.s_q + tok;
            float* dst0 = p.part_o + (prow_id * kHeads + row) * kDv + rank * kVcolsPerCta;
#pragma unroll 1
            for (int cc = 0; cc < 8; ++cc) {
              uint32_t r[32];
              tmem_ld32(tmem + lane_base + kColO + 32u * cc, r);
              tmem_wait_ld();
              float4* dst = reinterpret_cast<float4*>(dst0 + 32 * cc);
#pragma unroll
              for (int k = 0; k < 8; ++k)
                dst[k] = make_float4(__uint_as_float(r[4 * k]) * inv, __uint_as_float(r[4 * k + 1]) * inv,
                                     __uint_as_float(r[4 * k + 2]) * inv, __uint_as_float(r[4 * k + 3]) * inv);
            }
            if (rank == 0) p.part_lse[prow_id * kHeads + row] = lse;
          }
          tc_fence_before();
          mbar_arrive(bar(kOFree));
        }
      }
      ++nseg;
    }
  } else if (warp == 4) {
    // ===================================================== MMA issuer
    if (lane == 0) {
      SegIter it(p, unit);
      Seg sg;
      uint32_t g = 0, nseg = 0;
      bool ok = true;
      auto issue_pv = [&](uint32_t gg, bool first) -> bool {
        const uint32_t pb = gg & 1u, ph = (gg >> 1) & 1u;
        if (!wait_bar<false>(bar(kPFull0 + pb), ph, ctl)) return false;
        if (first && !wait_bar<false>(bar(kOFree), (nseg & 1u) ^ 1u, ctl)) return false;
        tc_fence_after();
        const uint32_t stg = sKv + pb * kStageBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = smem_desc(sP + pb * kPBytes + 32u * kk, 16u, 1024u);
          const uint64_t bd = smem_desc(stg + 2048u * kk, 8192u, 1024u);  // V, MN-major
          umma_f16(tmem + kColO, ad, bd, kIdescPV, (first && kk == 0) ? 0u : 1u);
        }
        umma_commit(bar(kKvEmpty0 + pb));
        umma_commit(bar(kPFree0 + pb));
        return true;
      };
      while (ok && it.next(sg)) {
        if (!(ok = wait_bar<false>(bar(kQFull), nseg & 1u, ctl))) break;
        tc_fence_after();
        for (int j = sg.t0; j < sg.t1; ++j, ++g) {
          const uint32_t st = g & 1u, ph = (g >> 1) & 1u;
          if (!(ok = wait_bar<false>(bar(kKvFull0 + st), ph, ctl))) break;
          if (!(ok = wait_bar<false>(bar(kSFree0 + st), ph ^ 1u, ctl))) break;
          tc_fence_after();
          const uint32_t stg = sKv + st * kStageBytes;
          for (int c = 0; c < nq; ++c) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = smem_desc(sQ + c * kQChunkBytes + 32u * kk, 16u, 1024u);
              const uint64_t bd = smem_desc(stg + c * kKvChunkBytes + 32u * kk, 16u, 1024u);
              umma_f16(tmem + kColS + 64u * st, ad, bd, kIdescQK, (c | kk) != 0 ? 1u : 0u);
            }
          }
          umma_commit(bar(kSFull0 + st));
          if (j == sg.t1 - 1) umma_commit(bar(kQEmpty));
          if (j > sg.t0 && !(ok = issue_pv(g - 1u, j - 1 == sg.t0))) break;
        }
        if (!ok) break;
        if (!(ok = issue_pv(g - 1u, sg.t1 - 1 == sg.t0))) break;
        umma_commit(bar(kOFull));
        ++nseg;
      }
      // every MMA issued so far is complete before TMEM is released
      umma_commit(bar(kMmaDone));
      drain_bar(bar(kMmaDone), 0);
    }
    __syncwarp();
  } else {
    // ===================================================== loads
    const int ptid = threadIdx.x - 160;  // 0..127
    if (!kSparse) {
      if (ptid == 0) {
        SegIter it(p, unit);
        Seg sg;
        uint32_t g = 0, nseg = 0;
        bool ok = true;
        uint32_t last_q = 0xffffffffu;
        while (ok && it.next(sg)) {
          if (!(ok = wait_bar<false>(bar(kQEmpty), (nseg & 1u) ^ 1u, ctl))) break;
          mbar_arrive_expect_tx(bar(kQFull), nq * kQChunkBytes);
          const int qy = (sg.b * p.s_q + tok) * kHeads;
          for (int c = 0; c < nq; ++c)
            tma_load_2d(sQ + c * kQChunkBytes, &tm_q, (chunk0 + c) * kChunk, qy, bar(kQFull));
          last_q = nseg;
          const int* bt_row = p.block_table + static_cast<long long>(sg.b) * p.bt_stride;
          for (int j = sg.t0; j < sg.t1; ++j, ++g) {
            const uint32_t st = g & 1u, ph = (g >> 1) & 1u;
            if (!(ok = wait_bar<false>(bar(kKvEmpty0 + st), ph ^ 1u, ctl))) break;
            int page = j < p.bt_stride ? bt_row[j] : -1;
            // an entry outside the pool reads the TMA fill value (zeros)
            const int y = (page >= 0 && page < p.num_pages) ? page * kPage
                                                             : static_cast<int>(p.num_pages) * kPage;
            mbar_arrive_expect_tx(bar(kKvFull0 + st), nq * kKvChunkBytes);
            for (int c = 0; c < nq; ++c)
              tma_load_2d(sKv + st * kStageBytes + c * kKvChunkBytes, &tm_kv, (chunk0 + c) * kChunk, y,
                          bar(kKvFull0 + st));
          }
          ++nseg;
        }
        if (!ok) {  // let copies in flight land before the CTA goes away
          if (last_q != 0xffffffffu) drain_bar(bar(kQFull), last_q & 1u);
          if (g >= 1) drain_bar(bar(kKvFull0 + ((g - 1) & 1u)), ((g - 1) >> 1) & 1u);
          if (g >= 2) drain_bar(bar(kKvFull0 + ((g - 2) & 1u)), ((g - 2) >> 1) & 1u);
        }
      }
    } else {
      // sparse gather: warp pw fills rows pw*16 .. pw*16+15 of each tile
      const int pw = ptid >> 5;
      SegIter it(p, unit);
      Seg sg;
      uint32_t g = 0, nseg = 0;
      bool ok = true;
      uint32_t last_q = 0xffffffffu;
      while (ok && it.next(sg)) {
        if (pw == 0) {  // warp-uniform outcome: the loader warps use warp-collective ops
          bool qok = true;
          if (lane == 0) {
            qok = wait_bar<false>(bar(kQEmpty), (nseg & 1u) ^ 1u, ctl);
            if (qok) {
              mbar_arrive_expect_tx(bar(kQFull), nq * kQChunkBytes);
              const int qy = (sg.b * p.s_q + tok) * kHeads;
              for (int c = 0; c < nq; ++c)
                tma_load_2d(sQ + c * kQChunkBytes, &tm_q, (chunk0 + c) * kChunk, qy, bar(kQFull));
              last_q = nseg;
            }
          }
          if (!(ok = __all_sync(0xffffffffu, qok))) break;
        }
        const int L = max(p.cache_lens[sg.b], 0);
        const int* idx = p.topk_idx + (static_cast<long long>(sg.b) * p.s_q + tok) * p.topk;
        const int* bt_row = p.block_table + static_cast<long long>(sg.b) * p.bt_stride;
        for (int j = sg.t0; j < sg.t1; ++j, ++g) {
          const uint32_t st = g & 1u, ph = (g >> 1) & 1u;
          if (!(ok = __all_sync(0xffffffffu, wait_bar<false>(bar(kKvEmpty0 + st), ph ^ 1u, ctl))))
            break;
          long long prow = -1;
          {
            const int pos = j * 64 + pw * 16 + (lane & 15);
            if (lane < 16 && pos < p.topk) {
              const int ix = idx[pos];
              if (ix >= 0 && ix < L && (ix >> 6) < p.bt_stride) {
                const int pg = bt_row[ix >> 6];
                if (pg >= 0 && pg < p.num_pages) prow = static_cast<long long>(pg) * kPage + (ix & 63);
              }
            }
          }
          const uint32_t vbits = __ballot_sync(0xffffffffu, prow >= 0) & 0xffffu;
          if (lane == 0)
            *reinterpret_cast<volatile uint16_t*>(smem + kOffMask + 8 * st + 2 * pw) =
                static_cast<uint16_t>(vbits);
          const uint32_t stg = sKv + st * kStageBytes;
          // each lane moves 16-byte pieces; nq * 8 pieces per row
          for (int rr = 0; rr < 16; ++rr) {
            const int r = pw * 16 + rr;
            const long long pr = __shfl_sync(0xffffffffu, prow, rr);
            for (int c16 = lane; c16 < nq * 8; c16 += 32) {
              const uint32_t dst = stg + (c16 >> 3) * kKvChunkBytes + r * 128 +
                                   (((c16 & 7) ^ (r & 7)) << 4);
              if (pr >= 0) {
                const uint4 v = *reinterpret_cast<const uint4*>(
                    p.kv + pr * kDqk + (chunk0 + (c16 >> 3)) * kChunk + (c16 & 7) * 8);
                st_shared_v4(dst, v.x, v.y, v.z, v.w);
              } else {
                st_shared_zero16(dst);
              }
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(bar(kKvFull0 + st));
        }
        ++nseg;
      }
      if (!ok && ptid == 0 && last_q != 0xffffffffu) drain_bar(bar(kQFull), last_q & 1u);
    }
  }

  // ======================================================= teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer no longer touches this CTA's shared memory
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
int decode_smem_bytes() { return kSmemBytes; }
int decode_threads() { return kNumThreads; }

cudaError_t decode_set_attrs() {
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mla_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

static void cluster_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int num_clusters,
                           cudaStream_t stream) {
  cfg = cudaLaunchConfig_t{};
  cfg.gridDim = dim3(2 * num_clusters, 1, 1);
  cfg.blockDim = dim3(kNumThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;  // the kernel always runs as CTA pairs
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
}

// Co-resident 2-CTA clusters of the decode kernel on the current device.
cudaError_t decode_max_clusters(int* n, int num_clusters_hint) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  cluster_config(cfg, attr, num_clusters_hint, nullptr);
  return cudaOccupancyMaxActiveClusters(n, mla_decode_kernel<false>, &cfg);
}

cudaError_t decode_launch(bool sparse, int num_clusters, cudaStream_t stream, const DecodeParams& p,
                          const CUtensorMap& tm_q, const CUtensorMap& tm_kv) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  cluster_config(cfg, attr, num_clusters, stream);
  return sparse ? cudaLaunchKernelEx(&cfg, mla_decode_kernel<true>, p, tm_q, tm_kv)
                : cudaLaunchKernelEx(&cfg, mla_decode_kernel<false>, p, tm_q, tm_kv);
}

}  // namespace mla
