// noalloc.cu — a decode step that allocates nothing: its workspace is a
// file-scope device array.
//
// Who needs it: callers that cannot call cudaMalloc when a decode step runs,
// for instance a serving runtime that captures its per-token work into a CUDA
// graph (device allocation is not allowed while a stream is being captured),
// or a host program that owns a fixed device-memory budget and forbids any
// allocation after start-up.  They call mla_decode_noalloc and pass only
// inputs and outputs.
//
// The array below is part of the library's device image: every GPU that loads
// the library holds it until the process exits.  Host code cannot pass the
// array's name to a kernel (on the host it is only a stand-in symbol), so the
// first call on each device looks its device address up with
// cudaGetSymbolAddress while that device is current, and later calls reuse it.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "mla_decode.h"

namespace {

constexpr size_t kScratchBytes = size_t(48) << 20;  // 48 MiB

static __device__ __align__(256) unsigned char g_mla_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  std::once_flag once;
  int status = MLA_OK;
  void* ptr = nullptr;
};
ScratchSlot g_slot[kMaxDevices];

// Device address of g_mla_scratch on the current device (looked up once).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_DEVICE;
  ScratchSlot& s = g_slot[dev];
  std::call_once(s.once, [&s] {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_mla_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      s.status = MLA_ERR_CUDA;
      return;
    }
    s.ptr = p;
  });
  *out = s.ptr;
  return s.status;
}

}  // namespace

extern "C" int mla_decode_noalloc(const void* q, const void* kv_cache, int64_t num_pages,
                                  const int32_t* block_table, int64_t bt_stride, const int32_t* cache_lens,
                                  int batch, int s_q, int num_heads, float softmax_scale,
                                  const int32_t* topk_idx, int topk, unsigned flags, void* out, float* lse,
                                  mla_stream_t stream) {
  // every argument check of mla_decode first: a rejected call leaves the
  // array (and the status word an earlier call left there) untouched
  int rc = mla::check_decode_args(q, kv_cache, num_pages, block_table, bt_stride, cache_lens, batch, s_q,
                                  num_heads, softmax_scale, topk_idx, topk, flags, out, lse);
  if (rc != MLA_OK) return rc;
  // the same number of work units the allocating path would use, fewer if
  // the workspace would not fit the array; reject what does not fit at all
  int err = MLA_OK;
  int units = mla_default_num_units(s_q, &err);
  if (units <= 0) return err != MLA_OK ? err : MLA_ERR_DEVICE;
  while (units > 1 && mla::ws_layout(batch, s_q, units).total > kScratchBytes) --units;
  const size_t need = mla::ws_layout(batch, s_q, units).total;
  if (need > kScratchBytes) return MLA_ERR_WORKSPACE;
  void* ws = nullptr;
  if ((rc = scratch_address(&ws)) != MLA_OK) return rc;
  // nothing in the array must start at zero: the plan rewrites every metadata
  // word and the status, partials are written before they are read
  if ((rc = mla_decode_plan(cache_lens, batch, s_q, topk, units, ws, kScratchBytes, stream)) != MLA_OK) return rc;
  if ((rc = mla_decode(q, kv_cache, num_pages, block_table, bt_stride, cache_lens, batch, s_q, num_heads,
                       softmax_scale, topk_idx, topk, flags, units, ws, kScratchBytes, out, lse, stream)) !=
      MLA_OK)
    return rc;
  return mla_combine(ws, kScratchBytes, batch, s_q, num_heads, flags, units, out, lse, stream);
}

extern "C" int mla_noalloc_status(mla_stream_t stream) {
  void* ws = nullptr;
  const int rc = scratch_address(&ws);
  if (rc != MLA_OK) return rc;
  return mla_workspace_status(ws, stream);
}

extern "C" int mla_noalloc_workspace(void** dev_ptr, size_t* bytes) {
  if (!dev_ptr || !bytes) return MLA_ERR_INVALID_ARG;
  void* ws = nullptr;
  const int rc = scratch_address(&ws);
  if (rc != MLA_OK) return rc;
  *dev_ptr = ws;
  *bytes = kScratchBytes;
  return MLA_OK;
}
