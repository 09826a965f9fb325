// indexer_kernel.cu — the sparse-attention indexer: token scores over a
// request's paged index keys on tcgen05, then a radix top-k selection that
// writes the index lists the sparse decode consumes (include/mla_indexer.h).
//
// Score ("The 31-Millisecond Smoking Gun", the DeepSeek-V4-Flash architecture
// paragraph and the indexer passage, read as the published DSA form with 64
// index heads): I[b, t, j] = sum_h w[b, t, h] * ReLU(q_I[b, t, h] . k_I[j]).
//
//   mla_indexer_scores_kernel: CTA = (query token, 1024 positions), 192
//     threads, two CTAs per SM.  Warp 0 loads the token's 64 x 128 index
//     query once and 128-position tiles (two pages, 32 KiB) of index keys
//     through a 2-slot ring by TMA; warp 1 issues 8 MMAs of M128 (positions)
//     N64 (heads) K16 per tile into one of two TMEM accumulators; warps 2..5
//     (one position per thread) apply ReLU, weight and sum the 64 heads in
//     fp32 and store the score.  HBM-bound: 256 B of keys per position.
//   mla_topk_kernel: CTA = query token, 1024 threads.  Scores map to
//     order-preserving 32-bit keys; three histogram passes (11, 11, 10 bits;
//     per-warp histograms: keys of similar magnitude share their top bits and
//     would serialise on a few shared words) find the k-th largest key T and
//     how many keys equal to T to keep; a final ordered pass keeps every key
//     > T and the first of those == T (smaller positions) and writes them in
//     position order (one block scan per 32 positions per thread).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "kernel_common.cuh"
#include "mla_indexer.h"

namespace mla {
namespace {

constexpr int kIH = 64;                        // index heads (N)
constexpr int kID = 128;                       // index dims (K)
constexpr int kIRow = 128;                     // bytes per 128-byte swizzle row (64 bf16)
constexpr int kTileRows = 128;                 // positions per tile = two pages (M)
constexpr int kChunkTiles = 8;                 // tiles per CTA: 1024 positions
constexpr int kChunkPos = kChunkTiles * kTileRows;
constexpr int kISlots = 2;
constexpr int kITile = 2 * kTileRows * kIRow;  // 32 KiB: two 64-dim chunks of 128 rows
constexpr int kIQ = 2 * kIH * kIRow;           // 16 KiB: the index query, two 64-dim chunks
constexpr int kIOffQ = 0;
constexpr int kIOffRing = kIQ;
constexpr int kIOffBar = kIOffRing + kISlots * kITile;  // 80 KiB
constexpr int kINumBars = 1 + 2 * kISlots + 2 * 2 + 1;
constexpr int kSlack = 1024;
constexpr int kISmem = kIOffBar + kINumBars * 8 + 16 + kSlack;
constexpr int kIThreads = 192;
constexpr uint32_t kITmemCols = 128;           // two 64-column accumulators
constexpr uint32_t kIdescIdx = idesc_bf16(128, kIH, 0);
static_assert(2 * (kISmem + 1024) <= 233472, "two CTAs per SM");

struct IndexerParams {
  const float* w;  // [B * s_q, 64]
  const int* block_table;
  long long bt_stride;
  const int* cache_lens;
  float* scores;
  long long scores_stride;
  int s_q, causal, max_len;
  int* status;
};

// Visible positions of query token t of request b (lengths beyond max_len
// are clamped to it).
__device__ __forceinline__ int visible(const int* lens, int b, int t, int s_q, int causal, int max_len) {
  int L = lens[b];
  L = L < 0 ? 0 : (L > max_len ? max_len : L);
  int n = causal ? L - s_q + t + 1 : L;
  n = n > L ? L : n;
  return n > 0 ? n : 0;
}

__global__ void __launch_bounds__(kIThreads, 2)
mla_indexer_scores_kernel(const __grid_constant__ IndexerParams p, const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t mis = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + mis;
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bt = blockIdx.y;
  const int b = bt / p.s_q, t = bt - b * p.s_q;
  const int vis = visible(p.cache_lens, b, t, p.s_q, p.causal, p.max_len);
  const int p0 = blockIdx.x * kChunkPos;
  if (threadIdx.x == 0 && blockIdx.x == 0 && p.cache_lens[b] > p.max_len && t == 0)
    atomicCAS(p.status, 0, static_cast<int>(kStBadTable));
  if (p0 >= vis) return;  // the whole CTA: nothing of this chunk is visible
  const int ntiles = min(kChunkTiles, (vis - p0 + kTileRows - 1) / kTileRows);

  const uint32_t bar0 = sbase + kIOffBar;
  const uint32_t bar_q = bar0;
  auto full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto empty = [&](int s) { return bar0 + 8u * (1 + kISlots + s); };
  auto acc_full = [&](int s) { return bar0 + 8u * (1 + 2 * kISlots + s); };
  auto acc_empty = [&](int s) { return bar0 + 8u * (3 + 2 * kISlots + s); };
  const uint32_t bar_drain = bar0 + 8u * (kINumBars - 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kIOffBar + kINumBars * 8);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kIOffBar + kINumBars * 8 + 4);
  auto slot = [&](int s) { return sbase + static_cast<uint32_t>(kIOffRing + s * kITile); };

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < kISlots; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(acc_full(s), 1);
      mbar_init(acc_empty(s), 4);  // one arrival per epilogue warp
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kITmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  Ctl ctl;
  ctl.abort = abort_flag;
  ctl.n_remote = 0;
  ctl.status = p.status;

  int issued = 0;
  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      mbar_arrive_expect_tx(bar_q, kIQ);
      tma_load_2d(sbase + kIOffQ, &tm_q, 0, bt * kIH, bar_q);
      tma_load_2d(sbase + kIOffQ + kIQ / 2, &tm_q, 64, bt * kIH, bar_q);
      const int* table = p.block_table + static_cast<long long>(b) * p.bt_stride;
      for (int i = 0; i < ntiles; ++i) {
        const int s = i % kISlots;
        if (i >= kISlots && !wait_bar<false>(empty(s), ((i / kISlots) - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(full(s), kITile);
        const int page0 = (p0 + i * kTileRows) / kPage;
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          // a page past the table's used part reads as zeros (negative row)
          const int pg = page0 + pp;
          const int id = (static_cast<long long>(pg) * kPage < p.max_len) ? table[pg] : -1;
#pragma unroll
          for (int c = 0; c < 2; ++c)
            tma_load_2d(slot(s) + c * (kITile / 2) + pp * (kITile / 4), &tm_k, 64 * c, id * kPage, full(s));
        }
        issued = i + 1;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      bool ok = wait_bar<false>(bar_q, 0u, ctl);
      for (int i = 0; ok && i < ntiles; ++i) {
        const int s = i % kISlots, acc = i & 1;
        if (!(ok = wait_bar<false>(full(s), (i / kISlots) & 1, ctl))) break;
        if (i >= 2 && !(ok = wait_bar<false>(acc_empty(acc), ((i / 2) - 1) & 1, ctl))) break;
        tc_fence_after();
        const uint64_t ad = smem_desc(slot(s), 16u, 1024u);
        const uint64_t bd = smem_desc(sbase + kIOffQ, 16u, 1024u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_f16(tmem + static_cast<uint32_t>(acc * kIH),
                   ad + static_cast<uint64_t>(((kk >> 2) * (kITile / 2) + (kk & 3) * 32) >> 4),
                   bd + static_cast<uint64_t>(((kk >> 2) * (kIQ / 2) + (kk & 3) * 32) >> 4), kIdescIdx,
                   kk != 0 ? 1u : 0u);
        umma_commit(empty(s));
        umma_commit(acc_full(acc));
      }
      umma_commit(bar_drain);  // arrives once every MMA issued above has completed
    }
    __syncwarp();
  } else {
    // epilogue: warp w reads TMEM lanes 32 * (w % 4) .. +31 = those positions of the tile
    const int q4 = warp & 3;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    float wr[kIH];
#pragma unroll
    for (int h = 0; h < kIH; ++h) wr[h] = __ldg(p.w + static_cast<long long>(bt) * kIH + h);
    float* out = p.scores + static_cast<long long>(bt) * p.scores_stride;
    for (int i = 0; i < ntiles; ++i) {
      const int acc = i & 1;
      if (!warp_wait(acc_full(acc), (i / 2) & 1, ctl)) break;
      tc_fence_after();
      uint32_t lo[32], hi[32];
      tmem_ld32(tl + static_cast<uint32_t>(acc * kIH), lo);
      tmem_ld32(tl + static_cast<uint32_t>(acc * kIH + 32), hi);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(acc));
      float sc = 0.f;
#pragma unroll
      for (int h = 0; h < 32; ++h) sc = fmaf(wr[h], fmaxf(__uint_as_float(lo[h]), 0.f), sc);
#pragma unroll
      for (int h = 0; h < 32; ++h) sc = fmaf(wr[32 + h], fmaxf(__uint_as_float(hi[h]), 0.f), sc);
      const int pos = p0 + i * kTileRows + q4 * 32 + lane;
      if (pos < vis) out[pos] = sc + 0.f;  // + 0: a negative zero becomes +0
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 32) drain_bar(bar_drain, 0u);  // MMAs finish before TMEM is released
  if (threadIdx.x == 0 && *abort_flag) {           // loads in flight land before the CTA exits
    for (int i = issued > kISlots ? issued - kISlots : 0; i < issued; ++i)
      drain_bar(full(i % kISlots), (i / kISlots) & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kITmemCols);
  }
}

// ------------------------------------------------------------------ top-k
constexpr int kKThreads = 1024;
constexpr int kPer = 32;  // consecutive positions per thread and pass: 128 B of loads in flight
constexpr int kKSmem = 32 * 1024 * 4;  // per-warp histograms
// a warp counts at most kPer * 32 keys per span of kPer * kKThreads positions
constexpr int kMaxTopkLen = (65535 / (kPer * 32)) * kPer * kKThreads;  // 2,064,384 positions per row

// Scores j0 .. j0 + kPer - 1 of a row (0 past `vis`); the row's stride is a
// multiple of 4 floats, so whole runs load as four 16-byte loads.
__device__ __forceinline__ void load_run(const float* __restrict__ row, int j0, int vis, float (&v)[kPer]) {
  if (j0 + kPer <= vis) {
#pragma unroll
    for (int i = 0; i < kPer / 4; ++i) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(row + j0) + i);
      v[4 * i] = f.x;
      v[4 * i + 1] = f.y;
      v[4 * i + 2] = f.z;
      v[4 * i + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kPer; ++i) v[i] = j0 + i < vis ? __ldg(row + j0 + i) : 0.f;
  }
}

// Order-preserving key of a finite float (larger float -> larger key; the
// two zeros are one key).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum over the block of one value per thread (in thread
// order); *total receives the block's sum.  Uses warp_sums[32].
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  *total = warp_sums[31];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kKThreads)
mla_topk_kernel(const float* __restrict__ scores, long long stride, const int* __restrict__ lens, int s_q,
                int causal, int max_len, int topk, int* __restrict__ out) {
  // per-warp histograms, two 16-bit bins per word (a warp counts at most
  // kPer * 32 keys per span of kPer * 1024 positions, <= 65,535 for the
  // kMaxTopkLen positions the host admits, so the halves never carry);
  // merged into hist[] after each pass
  extern __shared__ uint32_t warp_hist[];  // [32][1024]
  __shared__ int hist[2048];
  __shared__ int warp_sums[32];
  __shared__ int s_digit, s_above;
  const int bt = blockIdx.x;
  const int b = bt / s_q, t = bt - b * s_q;
  const int vis = visible(lens, b, t, s_q, causal, max_len);
  const float* row = scores + static_cast<long long>(bt) * stride;
  int* o = out + static_cast<long long>(bt) * topk;
  const int tid = threadIdx.x;
  if (vis <= topk) {  // everything visible is selected
    for (int j = tid; j < topk; j += kKThreads) o[j] = j < vis ? j : -1;
    return;
  }

  // ---- the k-th largest key: 11 + 11 + 10 bits, most significant first
  uint32_t prefix = 0, mask = 0;
  int krem = topk;  // how many of the keys matching the prefix are still to be taken
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass == 2 ? 1024 : 2048;
    for (int i = tid; i < 32 * 1024; i += kKThreads) warp_hist[i] = 0u;
    __syncthreads();
    uint32_t* wh = warp_hist + (tid >> 5) * 1024;
    for (int base = 0; base < vis; base += kPer * kKThreads) {
      const int j0 = base + tid * kPer;
      float v[kPer];
      load_run(row, j0, vis, v);
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const uint32_t key = order_key(v[i]);
        const bool in = j0 + i < vis && (key & mask) == prefix;
        const uint32_t bin = in ? (key >> shift) & static_cast<uint32_t>(nb - 1) : 0xffffffffu;
        if (in) atomicAdd(&wh[bin >> 1], 1u << (16u * (bin & 1u)));
      }
    }
    __syncthreads();
    for (int bin = tid; bin < nb; bin += kKThreads) {
      int c = 0;
#pragma unroll 8
      for (int w = 0; w < 32; ++w) c += static_cast<int>((warp_hist[w * 1024 + (bin >> 1)] >> (16 * (bin & 1))) & 0xffffu);
      hist[bin] = c;
    }
    __syncthreads();
    // bins from the top: thread i holds bins nb-1-per*i .. (descending)
    const int per = nb / kKThreads;
    int mine = 0;
    for (int k = 0; k < per; ++k) mine += hist[nb - 1 - per * tid - k];
    int total = 0;
    const int above = block_exclusive_scan(mine, warp_sums, &total);
    if (above < krem && krem <= above + mine) {
      int acc = above;
      for (int k = 0; k < per; ++k) {
        const int bin = nb - 1 - per * tid - k;
        if (krem <= acc + hist[bin]) {
          s_digit = bin;
          s_above = acc;
          break;
        }
        acc += hist[bin];
      }
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(s_digit) << shift;
    mask |= static_cast<uint32_t>(nb - 1) << shift;
    krem -= s_above;
    __syncthreads();
  }
  const uint32_t T = prefix;  // keys > T are all taken, and the first krem keys == T

  // ---- ordered output, positions ascending: each thread owns kPer
  // consecutive positions of a block-wide span; one scan of the per-thread
  // counts places them
  int taken = 0, eq_seen = 0;
#pragma unroll 1
  for (int base = 0; base < vis; base += kPer * kKThreads) {
    const int j0 = base + tid * kPer;
    uint32_t gt = 0, eq = 0;  // bit i: position j0 + i
    float v[kPer];
    load_run(row, j0, vis, v);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      if (j0 + i < vis) {
        const uint32_t key = order_key(v[i]);
        gt |= static_cast<uint32_t>(key > T) << i;
        eq |= static_cast<uint32_t>(key == T) << i;
      }
    }
    int eq_total = 0;
    int eq_rank = eq_seen + block_exclusive_scan(__popc(eq), warp_sums, &eq_total);
    uint32_t sel = gt;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      if ((eq >> i) & 1u) {
        if (eq_rank < krem) sel |= 1u << i;
        ++eq_rank;
      }
    }
    int sel_total = 0;
    int at = taken + block_exclusive_scan(__popc(sel), warp_sums, &sel_total);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      if ((sel >> i) & 1u) {
        if (at < topk) o[at] = j0 + i;
        ++at;
      }
    }
    taken += sel_total;
    eq_seen += eq_total;
  }
}

// ------------------------------------------------------------------ host side
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

// A bf16 [rows, 128] tensor as boxes of {64 columns, 64 rows} in the 128-byte swizzle.
int encode_rows128(CUtensorMap* m, const void* base, uint64_t rows) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return MLA_ERR_CUDA;
  const cuuint64_t size[2] = {static_cast<cuuint64_t>(kID), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kID) * 2};
  const cuuint32_t box[2] = {64u, 64u};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), size, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_CUDA;
}

constexpr int kMaxDev = 64;
struct IndexerDevice {
  std::once_flag once;
  int status = MLA_OK;
};
IndexerDevice g_idx_dev[kMaxDev];

int indexer_device_ready() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return MLA_ERR_DEVICE;
  IndexerDevice& st = g_idx_dev[dev];
  std::call_once(st.once, [&st, dev] {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        major != 10 || minor != 3) {
      st.status = MLA_ERR_DEVICE;
      return;
    }
    if (cudaFuncSetAttribute(mla_indexer_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kISmem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(mla_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kKSmem) != cudaSuccess) {
      cudaGetLastError();
      st.status = MLA_ERR_CUDA;
    }
  });
  return st.status;
}

bool al(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int common_checks(const int32_t* cache_lens, int batch, int s_q, unsigned flags, int max_len, const float* scores,
                  int64_t scores_stride, const int* status) {
  if (!cache_lens || !scores || !status || !al(cache_lens, 4) || !al(scores, 16) || !al(status, 4))
    return MLA_ERR_INVALID_ARG;
  if (batch < 1 || max_len < 0 || (flags & ~static_cast<unsigned>(MLA_FLAG_CAUSAL)) != 0) return MLA_ERR_INVALID_ARG;
  if (s_q < 1 || s_q > MLA_MAX_SQ) return MLA_ERR_UNSUPPORTED;
  if (scores_stride < max_len || (scores_stride & 3) != 0) return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(batch) * s_q > 65535) return MLA_ERR_UNSUPPORTED;  // one grid row per query token
  return MLA_OK;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

int mla_indexer_scores(const void* q_idx, const float* w_idx, const void* k_idx_cache, int64_t num_pages,
                       const int32_t* block_table, int64_t bt_stride, const int32_t* cache_lens, int batch,
                       int s_q, unsigned flags, int max_len, float* scores, int64_t scores_stride, int* status,
                       mla_stream_t stream) {
  int rc = common_checks(cache_lens, batch, s_q, flags, max_len, scores, scores_stride, status);
  if (rc != MLA_OK) return rc;
  if (!q_idx || !w_idx || !k_idx_cache || !block_table || !al(q_idx, 16) || !al(w_idx, 4) ||
      !al(k_idx_cache, 16) || !al(block_table, 4))
    return MLA_ERR_INVALID_ARG;
  if (num_pages < 1 || num_pages > (INT32_MAX / kPage) - 1 || bt_stride < 1) return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_len) > 64 * bt_stride) return MLA_ERR_INVALID_ARG;
  if ((rc = indexer_device_ready()) != MLA_OK) return rc;
  if (max_len == 0) return MLA_OK;
  CUtensorMap tm_q, tm_k;
  if ((rc = encode_rows128(&tm_q, q_idx, static_cast<uint64_t>(batch) * s_q * kIH)) != MLA_OK ||
      (rc = encode_rows128(&tm_k, k_idx_cache, static_cast<uint64_t>(num_pages) * kPage)) != MLA_OK)
    return rc;
  IndexerParams p;
  p.w = w_idx;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.cache_lens = cache_lens;
  p.scores = scores;
  p.scores_stride = scores_stride;
  p.s_q = s_q;
  p.causal = (flags & MLA_FLAG_CAUSAL) ? 1 : 0;
  p.max_len = max_len;
  p.status = status;
  const dim3 grid((max_len + kChunkPos - 1) / kChunkPos, batch * s_q, 1);
  mla_indexer_scores_kernel<<<grid, kIThreads, kISmem, static_cast<cudaStream_t>(stream)>>>(p, tm_q, tm_k);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_topk(const float* scores, int64_t scores_stride, const int32_t* cache_lens, int batch, int s_q,
             unsigned flags, int max_len, int topk, int32_t* out_idx, int* status, mla_stream_t stream) {
  int rc = common_checks(cache_lens, batch, s_q, flags, max_len, scores, scores_stride, status);
  if (rc != MLA_OK) return rc;
  if (!out_idx || !al(out_idx, 4) || topk < 1 || topk > 65536) return MLA_ERR_INVALID_ARG;
  if (max_len > kMaxTopkLen) return MLA_ERR_UNSUPPORTED;
  if ((rc = indexer_device_ready()) != MLA_OK) return rc;
  mla_topk_kernel<<<batch * s_q, kKThreads, kKSmem, static_cast<cudaStream_t>(stream)>>>(
      scores, scores_stride, cache_lens, s_q, (flags & MLA_FLAG_CAUSAL) ? 1 : 0, max_len, topk, out_idx);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // extern "C"
