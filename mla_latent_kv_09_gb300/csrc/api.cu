// api.cu — host side of the C ABI declared in include/mla_decode.h:
// argument checks, device checks, TMA descriptor encoding and launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "mla_decode.h"
#include "plan.cuh"

namespace mla {
__global__ void mla_plan_kernel(const int* lens, int B, int topk, int tile_rows, int U, int* hdr,
                                int* unit_meta, int* req_meta, int slots_cap);
__global__ void mla_wait_timeout_kernel(int* status);
__global__ void mla_combine_kernel(const int* hdr, const int* req_meta, const float* part_lse,
                                   const uint16_t* part_o, int part_bf16, int s_q, int out_fp32, void* out,
                                   float* lse, int n_bt);
__global__ void mla_validate_kernel(const int* lens, const int* bt, long long bt_stride,
                                    long long num_pages, int B, int s_q, const int* topk_idx, int topk,
                                    const uint16_t* kv, int check_range, int* status);
int decode_smem_bytes();
int decode_threads(bool sparse, bool fp8);
cudaError_t decode_set_attrs();
cudaError_t decode_max_clusters(int* n, int num_clusters_hint);
cudaError_t decode_launch(bool sparse, bool fp8, bool pair_tiles, int num_clusters, cudaStream_t stream,
                          const DecodeParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kv,
                          const CUtensorMap& tm_rope);
cudaError_t mtp_set_attrs();
cudaError_t mtp_max_clusters(int* n, int num_clusters_hint);
cudaError_t mtp_launch(bool bf16_pv, int num_clusters, cudaStream_t stream, const DecodeParams& p,
                       const CUtensorMap& tm_q, const CUtensorMap& tm_k3, const CUtensorMap& tm_v2,
                       const CUtensorMap& tm_out, const CUtensorMap& tm_part);
}  // namespace mla

using namespace mla;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxUnits = 4096;

struct DeviceState {
  std::once_flag once;
  int status = MLA_OK;
  int max_clusters = 0;      // co-resident 2-CTA clusters of the one-token kernel
  int max_clusters_mtp = 0;  // co-resident 4-CTA clusters of the two-token kernel
};
DeviceState g_dev[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

// Checks that the current device is a compute capability 10.3 part and sets
// the decode kernels up for it (once per device).
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_DEVICE;
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_DEVICE;
  DeviceState& st = g_dev[dev];
  std::call_once(st.once, [&st, dev] {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      st.status = MLA_ERR_DEVICE;
      return;
    }
    if (major != 10 || minor != 3) {
      st.status = MLA_ERR_DEVICE;
      return;
    }
    if (decode_set_attrs() != cudaSuccess || mtp_set_attrs() != cudaSuccess) {
      cudaGetLastError();
      st.status = MLA_ERR_CUDA;
      return;
    }
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int n = 0;
    if (decode_max_clusters(&n, sms / 2 > 0 ? sms / 2 : 1) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = sms / 2;  // one cluster per SM pair
    }
    st.max_clusters = n > 0 ? n : 1;
    int n4 = 0;
    if (mtp_max_clusters(&n4, sms / 4 > 0 ? sms / 4 : 1) != cudaSuccess || n4 <= 0) {
      cudaGetLastError();
      n4 = sms / 4;
    }
    st.max_clusters_mtp = n4 > 0 ? n4 : 1;
  });
  *out = &st;
  return st.status;
}

int last_cuda_error() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int resolve_units(int s_q, int num_units, int* units) {
  if (num_units < 0 || num_units > kMaxUnits) return MLA_ERR_INVALID_ARG;
  if (num_units > 0) {
    *units = num_units;
    return MLA_OK;
  }
  int err = MLA_OK;
  const int u = mla_default_num_units(s_q, &err);
  if (u <= 0) return err != MLA_OK ? err : MLA_ERR_DEVICE;
  *units = u;
  return MLA_OK;
}

int encode_2d(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MLA_ERR_CUDA;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDqk), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDqk) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kChunk), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_CUDA;
}

// The cache as a 3-D tensor (x: column within a 64-column chunk, y: row,
// z: chunk): one box fetches `box_chunks` chunks of 64 rows in one request.
int encode_kv_3d(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_chunks) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MLA_ERR_CUDA;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kChunk), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(kNumChunks)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kDqk) * 2, static_cast<cuuint64_t>(kChunk) * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kChunk), static_cast<cuuint32_t>(kPage), box_chunks};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_CUDA;
}

// An FP8 cache (656-byte rows) for the one-token kernel: `lat` maps each row's
// first 528 bytes (512 E4M3 codes, the scale bytes) as 132 32-bit words, one
// 64-row box per tile, landing unswizzled; `rope` maps the row as 328 bf16
// elements, a box of 64 of them (the RoPE dims, from element 264 = byte 528)
// by 64 rows, 128B-swizzled like every chunk of the bf16 path.
int encode_fp8_kv(CUtensorMap* lat, CUtensorMap* rope, const void* base, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MLA_ERR_CUDA;
  const cuuint64_t strides[1] = {656};
  const cuuint32_t estr[2] = {1, 1};
  const cuuint64_t dl[2] = {164, static_cast<cuuint64_t>(rows)};
  const cuuint32_t bl[2] = {132, static_cast<cuuint32_t>(kPage)};
  CUresult r = fn(lat, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dl, strides, bl, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return MLA_ERR_CUDA;
  const cuuint64_t dr[2] = {328, static_cast<cuuint64_t>(rows)};
  const cuuint32_t br[2] = {static_cast<cuuint32_t>(kChunk), static_cast<cuuint32_t>(kPage)};
  r = fn(rope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dr, strides, br, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_CUDA;
}

// An output tensor of 512 columns per row (bf16 or fp32) for tensor stores of
// 32-row boxes of 64-byte rows (32 bf16 or 16 fp32 columns), staged with the
// 64-byte swizzle as the two-token kernel writes them.
int encode_out_2d(CUtensorMap* m, void* base, uint64_t rows, bool fp32) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MLA_ERR_CUDA;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDv), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDv) * (fp32 ? 4 : 2)};
  const cuuint32_t box[2] = {fp32 ? 16u : 32u, 32u};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base,
                        dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace

extern "C" {

int mla_default_num_units(int s_q, int* err) {
  DeviceState* st = nullptr;
  const int rc = device_state(&st);
  if (err) *err = rc;
  if (rc != MLA_OK) return 0;
  if (s_q < 1 || s_q > MLA_MAX_SQ) {
    if (err) *err = MLA_ERR_UNSUPPORTED;
    return 0;
  }
  // s_q = 2: one unit is a 4-CTA cluster serving both tokens (dense), or two
  // 2-CTA clusters, one per token (top-k); take what both can keep resident
  int u = st->max_clusters / s_q;
  if (s_q == 2 && st->max_clusters_mtp < u) u = st->max_clusters_mtp;
  return u > 0 ? (u < kMaxUnits ? u : kMaxUnits) : 1;
}

size_t mla_decode_workspace_size(int batch, int s_q, int num_heads, int num_units) {
  if (batch < 1 || s_q < 1 || s_q > MLA_MAX_SQ || num_heads != kHeads) return 0;
  int units = 0;
  if (resolve_units(s_q, num_units, &units) != MLA_OK) return 0;
  return ws_layout(batch, s_q, units).total;
}

int mla_decode_plan(const int32_t* cache_lens, int batch, int s_q, int topk, int num_units, void* workspace,
                    size_t ws_bytes, mla_stream_t stream) {
  if (!cache_lens || !workspace || batch < 1 || topk < 0) return MLA_ERR_INVALID_ARG;
  if (s_q < 1 || s_q > MLA_MAX_SQ) return MLA_ERR_UNSUPPORTED;
  if (!aligned(workspace, 256)) return MLA_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != MLA_OK) return rc;
  int U = 0;
  if ((rc = resolve_units(s_q, num_units, &U)) != MLA_OK) return rc;
  const WsLayout L = ws_layout(batch, s_q, U);
  if (ws_bytes < L.total) return MLA_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  // up to 128 requests (every decode batch the bench times) one 128-thread
  // CTA: its block scans meet at fewer warps (~1 us off each call)
  mla_plan_kernel<<<1, batch <= 128 ? 128 : 1024, 0, static_cast<cudaStream_t>(stream)>>>(
      cache_lens, batch, topk, plan_tile_rows(s_q, topk), U, reinterpret_cast<int*>(ws + L.hdr),
      reinterpret_cast<int*>(ws + L.units), reinterpret_cast<int*>(ws + L.reqs), L.slots);
  return last_cuda_error();
}

int mla_decode_plan_host(const int32_t* lens, int batch, int s_q, int topk, int num_units, int32_t* unit_meta,
                         int32_t* req_meta) {
  if (!lens || !unit_meta || !req_meta || batch < 1 || topk < 0 || num_units < 1 || num_units > kMaxUnits)
    return MLA_ERR_INVALID_ARG;
  if (s_q < 1 || s_q > MLA_MAX_SQ) return MLA_ERR_UNSUPPORTED;
  const int tile_rows = plan_tile_rows(s_q, topk);
  int total = 0;
  for (int b = 0; b < batch; ++b) {
    const int n = plan_tiles(lens[b] > 0 ? lens[b] : 0, topk, tile_rows);
    req_meta[4 * b + 0] = n;
    req_meta[4 * b + 3] = total;
    total += plan_cost(n);
  }
  const int W = plan_width(total, num_units);
  int slots = 0;
  for (int b = 0; b < batch; ++b) {
    const int ns = plan_n_splits(req_meta[4 * b + 3], req_meta[4 * b + 0], W, num_units);
    req_meta[4 * b + 1] = ns;
    req_meta[4 * b + 2] = slots;
    if (ns > 1) slots += ns;
  }
  auto prefix = [&](int b) { return req_meta[4 * b + 3]; };
  for (int u = 0; u < num_units; ++u) {
    const UnitInfo ui = plan_unit(u, W, total, batch, prefix);
    int32_t* m = unit_meta + 5 * u;
    m[0] = ui.begin_req; m[1] = ui.begin_tile; m[2] = ui.end_req; m[3] = ui.end_tile; m[4] = ui.first_split;
  }
  return slots <= 2 * num_units ? MLA_OK : MLA_ERR_WORKSPACE;
}

}  // extern "C"

// Host-side checks of mla_decode's arguments (shared with the allocation-free
// step, which runs them before it touches its workspace).
int mla::check_decode_args(const void* q, const void* kv_cache, int64_t num_pages, const int32_t* block_table,
                          int64_t bt_stride, const int32_t* cache_lens, int batch, int s_q, int num_heads,
                          float softmax_scale, const int32_t* topk_idx, int topk, unsigned flags, const void* out,
                          const float* lse) {
  if (!q || !kv_cache || !block_table || !cache_lens || !out || !lse) return MLA_ERR_INVALID_ARG;
  if (batch < 1 || num_pages < 1 || bt_stride < 1 || topk < 0) return MLA_ERR_INVALID_ARG;
  if ((topk_idx == nullptr) != (topk == 0)) return MLA_ERR_INVALID_ARG;
  if (flags & ~static_cast<unsigned>(MLA_FLAG_CAUSAL | MLA_FLAG_OUT_FP32 | MLA_FLAG_VALIDATE | MLA_FLAG_BF16_PV |
                                     MLA_FLAG_KV_FP8))
    return MLA_ERR_INVALID_ARG;
  if (num_heads != kHeads || s_q < 1 || s_q > MLA_MAX_SQ) return MLA_ERR_UNSUPPORTED;
  if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
      !aligned(block_table, 4) || !aligned(cache_lens, 4) || (topk_idx && !aligned(topk_idx, 4)))
    return MLA_ERR_INVALID_ARG;
  if (num_pages > (INT32_MAX / kPage) - 1) return MLA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(batch) * s_q * kHeads > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

extern "C" {

int mla_decode(const void* q, const void* kv_cache, int64_t num_pages, const int32_t* block_table,
               int64_t bt_stride, const int32_t* cache_lens, int batch, int s_q, int num_heads,
               float softmax_scale, const int32_t* topk_idx, int topk, unsigned flags, int num_units,
               void* workspace, size_t ws_bytes, void* out, float* lse, mla_stream_t stream) {
  int rc = check_decode_args(q, kv_cache, num_pages, block_table, bt_stride, cache_lens, batch, s_q, num_heads,
                                 softmax_scale, topk_idx, topk, flags, out, lse);
  if (rc != MLA_OK) return rc;
  if (!workspace || !aligned(workspace, 256)) return MLA_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != MLA_OK) return rc;
  int U = 0;
  if ((rc = resolve_units(s_q, num_units, &U)) != MLA_OK) return rc;
  const WsLayout L = ws_layout(batch, s_q, U);
  if (ws_bytes < L.total) return MLA_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // two query tokens over a dense bf16 cache: the paired-SM kernel; an FP8
  // cache runs the one-token kernel on the same plan (its 128-row tiles
  // split in two)
  const bool pair_plan = plan_tile_rows(s_q, topk) == 128;
  const bool pair_path = pair_plan && !(flags & MLA_FLAG_KV_FP8);

  if (flags & MLA_FLAG_VALIDATE) {
    // the check records the first problem in the workspace status word; the
    // attention and combine kernels then leave their outputs unwritten, and
    // mla_workspace_status reports the code (no host synchronisation here)
    int* status = reinterpret_cast<int*>(ws + L.hdr) + kHdrStatus;
    // the fp16 value product: bf16 values (1) or FP8 rows (2) below 65536
    const int check_range = (flags & MLA_FLAG_KV_FP8) ? 2 : (pair_path && (flags & MLA_FLAG_BF16_PV)) ? 0 : 1;
    mla_validate_kernel<<<batch < 1024 ? batch : 1024, 256, 0, s>>>(
        cache_lens, block_table, bt_stride, num_pages, batch, s_q, topk_idx, topk,
        static_cast<const uint16_t*>(kv_cache), check_range, status);
    if ((rc = last_cuda_error()) != MLA_OK) return rc;
  }

  DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const uint16_t*>(q);
  p.kv = static_cast<const uint16_t*>(kv_cache);
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.cache_lens = cache_lens;
  p.topk_idx = topk_idx;
  p.topk = topk;
  p.batch = batch;
  p.s_q = s_q;
  p.causal = (flags & MLA_FLAG_CAUSAL) && topk_idx == nullptr ? 1 : 0;
  p.num_pages = num_pages;
  p.scale_log2 = static_cast<float>(static_cast<double>(softmax_scale) * 1.4426950408889634);
  p.out = out;
  p.lse = lse;
  p.out_fp32 = (flags & MLA_FLAG_OUT_FP32) ? 1 : 0;
  p.num_units = U;
  p.ws_hdr = reinterpret_cast<int*>(ws + L.hdr);
  p.unit_meta = reinterpret_cast<const int*>(ws + L.units);
  p.req_meta = reinterpret_cast<const int*>(ws + L.reqs);
  p.part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  p.part_o = reinterpret_cast<uint16_t*>(ws + L.part_o);
  p.part_bf16 = (flags & MLA_FLAG_BF16_PV) ? 1 : 0;

  // the two-token kernel moves Q through its 8 KiB chunk slots: 64-row boxes
  const bool fp8 = (flags & MLA_FLAG_KV_FP8) != 0;
  CUtensorMap tm_q, tm_kv, tm_rope;
  if ((rc = encode_2d(&tm_q, q, static_cast<uint64_t>(batch) * s_q * kHeads, pair_path ? kPage : kHeads)) !=
      MLA_OK)
    return rc;
  if (fp8) {
    if ((rc = encode_fp8_kv(&tm_kv, &tm_rope, kv_cache, static_cast<uint64_t>(num_pages) * kPage)) != MLA_OK)
      return rc;
  } else {
    // one-token kernel: a page's nine chunks (S side) / eight value chunks (O
    // side) as one 3-D box each; the two-token kernel encodes its own maps
    const uint64_t rows = static_cast<uint64_t>(num_pages) * kPage;
    if ((rc = encode_kv_3d(&tm_kv, kv_cache, rows, kNumChunks)) != MLA_OK) return rc;
    if ((rc = encode_kv_3d(&tm_rope, kv_cache, rows, 8)) != MLA_OK) return rc;
  }

  // two query tokens, dense: both tokens share every tile (4-CTA clusters,
  // paired-SM MMAs); otherwise one 2-CTA cluster per (unit, token)
  cudaError_t e;
  if (pair_path) {
    CUtensorMap tm_k3, tm_v2;  // K: three chunks (a slot group) per load; V: two chunks per load
    const uint64_t rows = static_cast<uint64_t>(num_pages) * kPage;
    if ((rc = encode_kv_3d(&tm_k3, kv_cache, rows, 3)) != MLA_OK) return rc;
    if ((rc = encode_kv_3d(&tm_v2, kv_cache, rows, 2)) != MLA_OK) return rc;
    CUtensorMap tm_out, tm_part;  // O (bf16 or fp32) and the 16-bit partials, for the epilogue's tensor stores
    if ((rc = encode_out_2d(&tm_out, out, static_cast<uint64_t>(batch) * s_q * kHeads, p.out_fp32 != 0)) != MLA_OK)
      return rc;
    if ((rc = encode_out_2d(&tm_part, p.part_o, static_cast<uint64_t>(L.slots) * s_q * kHeads, false)) != MLA_OK)
      return rc;
    e = mtp_launch((flags & MLA_FLAG_BF16_PV) != 0, U, s, p, tm_q, tm_k3, tm_v2, tm_out, tm_part);
  } else {
    e = decode_launch(topk_idx != nullptr, fp8, pair_plan, U * s_q, s, p, tm_q, tm_kv, tm_rope);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

int mla_combine(void* workspace, size_t ws_bytes, int batch, int s_q, int num_heads, unsigned flags,
                int num_units, void* out, float* lse, mla_stream_t stream) {
  if (!workspace || !out || !lse || batch < 1) return MLA_ERR_INVALID_ARG;
  if (flags & ~static_cast<unsigned>(MLA_FLAG_CAUSAL | MLA_FLAG_OUT_FP32 | MLA_FLAG_VALIDATE | MLA_FLAG_BF16_PV |
                                     MLA_FLAG_KV_FP8))
    return MLA_ERR_INVALID_ARG;
  if (num_heads != kHeads || s_q < 1 || s_q > MLA_MAX_SQ) return MLA_ERR_UNSUPPORTED;
  if (!aligned(out, 16) || !aligned(lse, 4) || !aligned(workspace, 256)) return MLA_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != MLA_OK) return rc;
  int U = 0;
  if ((rc = resolve_units(s_q, num_units, &U)) != MLA_OK) return rc;
  const WsLayout L = ws_layout(batch, s_q, U);
  if (ws_bytes < L.total) return MLA_ERR_WORKSPACE;
  const char* ws = static_cast<const char*>(workspace);
  // a programmatic dependent of the decode kernel: scheduled while the decode
  // kernel's last units finish, it waits for that grid before reading
  cudaLaunchConfig_t cfg = {};
  // at most one wave: 76 x 16 blocks of 256 threads (8 per SM on 152 SMs),
  // each block taking every 76th (request, token) row
  cfg.gridDim = dim3(batch * s_q < 76 ? batch * s_q : 76, kHeads / 8, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, mla_combine_kernel, reinterpret_cast<const int*>(ws + L.hdr),
                         reinterpret_cast<const int*>(ws + L.reqs),
                         reinterpret_cast<const float*>(ws + L.part_lse),
                         reinterpret_cast<const uint16_t*>(ws + L.part_o), (flags & MLA_FLAG_BF16_PV) ? 1 : 0, s_q,
                         (flags & MLA_FLAG_OUT_FP32) ? 1 : 0, out, lse, batch * s_q);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

int mla_selftest_wait_timeout(void* workspace, size_t ws_bytes, mla_stream_t stream) {
  if (!workspace || ws_bytes < 256 || !aligned(workspace, 256)) return MLA_ERR_INVALID_ARG;
  int* status = static_cast<int*>(workspace) + kHdrStatus;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return MLA_ERR_CUDA;
  mla_wait_timeout_kernel<<<1, 32, 0, s>>>(status);
  return last_cuda_error();
}

int mla_workspace_status(const void* workspace, mla_stream_t stream) {
  if (!workspace) return MLA_ERR_INVALID_ARG;
  int h = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&h, static_cast<const int*>(workspace) + kHdrStatus, sizeof(int), cudaMemcpyDeviceToHost,
                      s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MLA_ERR_CUDA;
  return h;
}

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG: null pointer, bad size or misaligned buffer";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: shape or mode not supported (128 heads, 576/512 dims, s_q 1..8)";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace too small";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA: a CUDA call failed";
    case MLA_ERR_DEVICE: return "MLA_ERR_DEVICE: current device is not compute capability 10.3";
    case MLA_ERR_BAD_TABLE: return "MLA_ERR_BAD_TABLE: cache length or block-table entry out of range";
    case MLA_ERR_BAD_INDEX: return "MLA_ERR_BAD_INDEX: top-k index outside [-1, cache length)";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT: a device-side wait ran out";
    case MLA_ERR_VALUE_RANGE: return "MLA_ERR_VALUE_RANGE: a visible value dim is not finite or too large for fp16";
    default: return "unknown mla_status";
  }
}

}  // extern "C"
