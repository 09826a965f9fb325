// absorb_kernel.cu — the weight-absorption batched GEMMs on either side of
// absorbed-MLA decode ("DeepSeek V3/R1 Inference Efficiency (2)", §2.4.1,
// Compute: QKV projection Q''' = bmm(Q'', W_UK^T) and O projection
// O' = bmm(PV, W_UV)), and their C ABI (include/mla_absorb.h).
//
// Both are one small GEMM per head: M = the step's tokens (tiles of 128, the
// MMA's M), K and N from {128, 512}.  At decode batch sizes the weights
// (16 MiB each for 128 heads) dominate the bytes, so both kernels are bound
// by HBM: the design goal is every byte read once, loads in flight from the
// first cycle, and two CTAs per SM so that one CTA's epilogue overlaps the
// other's loads.  Operands arrive by TMA in the 128-byte swizzle the tensor
// cores read, products accumulate in TMEM (tcgen05.mma kind::f16, issued by
// one thread), and the epilogue goes TMEM -> registers -> bf16 -> swizzled
// shared memory -> TMA tensor store.
//
//   query side: CTA = (token tile, head, half of the 512 latent dims).
//     A = q_nope tile  [128 tokens x 128 d]      2 chunks of 64 d, 16 KiB each
//     B = W_UK[h] rows [256 c x 128 d], K-major 2 chunks of 64 d, 32 KiB each
//     8 MMAs of M128 N256 K16 into 256 TMEM columns; the RoPE dims are
//     copied by warps 1..3 of the upper-half CTA while the loads fly.
//   output side: CTA = (token tile, head, half of the 128 output dims).
//     K = 512 latent dims in 8 stages of 64 through a ring of 4 slots:
//     A = O tile [128 tokens x 64 c] 16 KiB, B = W_UV[h] [64 c x 64 d]
//     (MN-major: d contiguous) 8 KiB; 32 MMAs of M128 N64 K16.
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

constexpr int kAbsThreads = 128;  // four warps = TMEM lanes 0..127 = the tile's token rows
constexpr int kTokTile = 128;
constexpr int kDNope = 128;       // d
constexpr int kLatent = 512;      // c
constexpr int kRope = 64;
constexpr int kMaxAbsorbHeads = 128;
constexpr int kRowBytes = 128;    // one swizzle-atom row: 64 bf16
constexpr int kSlack = 1024;      // dynamic shared memory is re-aligned to 1024 B (128-byte swizzle atoms)

// ---- query side
constexpr int kQCols = 256;                        // latent dims per CTA (N)
constexpr int kQAChunk = kTokTile * kRowBytes;     // 16 KiB
constexpr int kQBChunk = kQCols * kRowBytes;       // 32 KiB
constexpr int kQOffA = 0;
constexpr int kQOffB = 2 * kQAChunk;               // also the output staging (4 x 16 KiB)
constexpr int kQOffBar = kQOffB + 2 * kQBChunk;    // 96 KiB
constexpr int kQSmem = kQOffBar + 64 + kSlack;
constexpr uint32_t kQTmemCols = 256;
constexpr uint32_t kIdescQ = idesc_bf16(128, kQCols, 0);

// ---- output side
constexpr int kOCols = 64;                         // output dims per CTA (N)
constexpr int kOKStage = 64;                       // latent dims per stage (K)
constexpr int kOStages = kLatent / kOKStage;       // 8
constexpr int kOSlots = 4;
constexpr int kOAChunk = kTokTile * kRowBytes;     // 16 KiB
constexpr int kOBChunk = kOKStage * kRowBytes;     // 8 KiB
constexpr int kOSlotBytes = kOAChunk + kOBChunk;   // 24 KiB
constexpr int kOOffBar = kOSlots * kOSlotBytes;    // 96 KiB
constexpr int kOSmem = kOOffBar + 128 + kSlack;
constexpr uint32_t kOTmemCols = 64;
constexpr uint32_t kIdescO = idesc_bf16(128, kOCols, 1);

static_assert(kQSmem <= 116 * 1024 && kOSmem <= 116 * 1024, "two CTAs per SM");

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
__global__ void __launch_bounds__(kAbsThreads, 2)
mla_absorb_q_kernel(const __grid_constant__ AbsorbParams p, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_out) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t mis = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + mis;
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kTokTile, h = blockIdx.y, half = blockIdx.z;
  const int c0 = half * kQCols;
  const uint32_t bar_full = sbase + kQOffBar;  // two: one per 64-dim K chunk
  const uint32_t bar_mma = bar_full + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kQOffBar + 24);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kQOffBar + 28);

  if (threadIdx.x == 0) {
    mbar_init(bar_full, 1);
    mbar_init(bar_full + 8, 1);
    mbar_init(bar_mma, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kQTmemCols);
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

  if (warp == 0) {
    if (lane == 0) {
      // loads for both K chunks first, then the MMAs as each chunk lands
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint32_t bar = bar_full + 8u * k;
        mbar_arrive_expect_tx(bar, kQAChunk + kQBChunk);
        tma_load_3d(sbase + kQOffA + k * kQAChunk, &tm_q, 64 * k, h, t0, bar);
        tma_load_2d(sbase + kQOffB + k * kQBChunk, &tm_w, 64 * k, h * kLatent + c0, bar);
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (!wait_bar<false>(bar_full + 8u * k, 0u, ctl)) break;
        tc_fence_after();
        const uint64_t ad = smem_desc(sbase + kQOffA + k * kQAChunk, 16u, 1024u);
        const uint64_t bd = smem_desc(sbase + kQOffB + k * kQBChunk, 16u, 1024u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_f16(tmem, ad + static_cast<uint64_t>((32 * kk) >> 4), bd + static_cast<uint64_t>((32 * kk) >> 4),
                   kIdescQ, (k | kk) != 0 ? 1u : 0u);
      }
      umma_commit(bar_mma);  // arrives once every MMA issued above has completed
    }
    __syncwarp();
  } else if (half == 1 && p.q_pe != nullptr) {
    // RoPE dims pass through unchanged: one 128-byte row per thread
    for (int r = threadIdx.x - 32; r < kTokTile; r += kAbsThreads - 32) {
      const int t = t0 + r;
      if (t >= p.num_tokens) break;
      const long long row = static_cast<long long>(t) * p.num_heads + h;
      const uint16_t* src = p.q_pe + row * p.in_stride;
      uint16_t* dst = p.out + row * p.out_stride + kLatent;
      uint4 v[kRope / 8];
#pragma unroll
      for (int i = 0; i < kRope / 8; ++i) v[i] = ld_global_nc_v4(src + 8 * i);
#pragma unroll
      for (int i = 0; i < kRope / 8; ++i) st_global_v4(dst + 8 * i, v[i]);
    }
  }

  // epilogue: four 64-column slices, each stored as soon as all rows are staged
  bool ok = warp_wait(bar_mma, 0u, ctl) && *abort_flag == 0u;
  tc_fence_after();
  const int row = warp * 32 + lane;
  const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
  for (int j = 0; j < kQCols / 64; ++j) {
    const uint32_t stage = sbase + kQOffB + j * kQAChunk;
    if (ok) {
      stage_slice(tl + 64u * j, stage, row);
      fence_proxy_async_smem();
    }
    ok = named_bar_all(1, kAbsThreads, ok);
    if (!ok) break;
    if (threadIdx.x == 0) {
      tma_store_3d(&tm_out, stage, c0 + 64 * j, h, t0);
      bulk_commit();
    }
  }
  if (threadIdx.x == 0) {
    bulk_wait_read();  // the staging tiles stay valid until the stores have read them
    if (*abort_flag) {  // teardown after a wait ran out: let copies and MMAs in flight finish
      drain_bar(bar_full, 0u);
      drain_bar(bar_full + 8, 0u);
      drain_bar(bar_mma, 0u);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kQTmemCols);
  }
}

// ============================================================ output side
__global__ void __launch_bounds__(kAbsThreads, 2)
mla_absorb_o_kernel(const __grid_constant__ AbsorbParams p, const __grid_constant__ CUtensorMap tm_o,
                    const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_out) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t mis = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + mis;
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kTokTile, h = blockIdx.y, d0 = blockIdx.z * kOCols;
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
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kOTmemCols);
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

  auto slot_a = [&](int s) { return sbase + static_cast<uint32_t>(s * kOSlotBytes); };
  auto slot_b = [&](int s) { return sbase + static_cast<uint32_t>(s * kOSlotBytes + kOAChunk); };

  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      for (int s = 0; s < kOStages; ++s) {
        const int slot = s % kOSlots;
        if (s >= kOSlots && !wait_bar<false>(bar_empty + 8 * slot, ((s / kOSlots) - 1) & 1, ctl)) break;
        const uint32_t bar = bar_full + 8 * slot;
        mbar_arrive_expect_tx(bar, kOSlotBytes);
        tma_load_3d(slot_a(slot), &tm_o, kOKStage * s, h, t0, bar);
        tma_load_2d(slot_b(slot), &tm_w, d0, h * kLatent + kOKStage * s, bar);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
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
      umma_commit(bar_mma);
    }
    __syncwarp();
  }

  bool ok = warp_wait(bar_mma, 0u, ctl) && *abort_flag == 0u;
  tc_fence_after();
  const uint32_t stage = slot_a(0);  // free once every MMA has completed
  if (ok) {
    stage_slice(tmem + (static_cast<uint32_t>(warp * 32) << 16), stage, warp * 32 + lane);
    fence_proxy_async_smem();
  }
  ok = named_bar_all(1, kAbsThreads, ok);
  if (threadIdx.x == 0) {
    if (ok) {
      tma_store_3d(&tm_out, stage, d0, h, t0);
      bulk_commit();
      bulk_wait_read();
    } else {
      for (int i = 0; i < kOSlots; ++i) drain_bar(bar_full + 8 * i, (((kOStages - 1 - i) / kOSlots)) & 1);
      drain_bar(bar_mma, 0u);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
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
    }
  });
  return st.status;
}

// A token-major activation [T, H, dims] with rows `stride` elements apart,
// as 3-D boxes of {64 dims, 1 head, 128 tokens} in the 128-byte swizzle.
int encode_act(CUtensorMap* m, const void* base, uint64_t dims, int64_t stride, int heads, int tokens) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return MLA_ERR_CUDA;
  const cuuint64_t size[3] = {dims, static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(tokens)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(stride) * 2,
                                 static_cast<cuuint64_t>(stride) * 2 * static_cast<cuuint64_t>(heads)};
  const cuuint32_t box[3] = {64u, 1u, static_cast<cuuint32_t>(kTokTile)};
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
  if ((rc = encode_act(&tm_q, q_nope, kDNope, q_stride, num_heads, num_tokens)) != MLA_OK ||
      (rc = encode_weight(&tm_w, w_uk, num_heads, kQCols)) != MLA_OK ||
      (rc = encode_act(&tm_out, out, kLatent, out_stride, num_heads, num_tokens)) != MLA_OK)
    return rc;
  AbsorbParams p;
  p.q_pe = static_cast<const uint16_t*>(q_pe);
  p.in_stride = q_stride;
  p.out = static_cast<uint16_t*>(out);
  p.out_stride = out_stride;
  p.num_tokens = num_tokens;
  p.num_heads = num_heads;
  p.status = status;
  const dim3 grid((num_tokens + kTokTile - 1) / kTokTile, num_heads, kLatent / kQCols);
  mla_absorb_q_kernel<<<grid, kAbsThreads, kQSmem, static_cast<cudaStream_t>(stream)>>>(p, tm_q, tm_w, tm_out);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
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
  if ((rc = encode_act(&tm_o, o, kLatent, o_stride, num_heads, num_tokens)) != MLA_OK ||
      (rc = encode_weight(&tm_w, w_uv, num_heads, kOKStage)) != MLA_OK ||
      (rc = encode_act(&tm_out, out, kDNope, out_stride, num_heads, num_tokens)) != MLA_OK)
    return rc;
  AbsorbParams p = {};
  p.num_tokens = num_tokens;
  p.num_heads = num_heads;
  p.status = status;
  const dim3 grid((num_tokens + kTokTile - 1) / kTokTile, num_heads, kDNope / kOCols);
  mla_absorb_o_kernel<<<grid, kAbsThreads, kOSmem, static_cast<cudaStream_t>(stream)>>>(p, tm_o, tm_w, tm_out);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // extern "C"
