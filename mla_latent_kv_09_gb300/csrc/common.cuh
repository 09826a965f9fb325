// common.cuh — constants, workspace layout and kernel parameter blocks shared
// by the device kernels and the host API of the MLA decode library.
#pragma once
#include <cstddef>
#include <cstdint>

namespace mla {

constexpr int kHeads = 128;   // query heads per token (M of every MMA)
constexpr int kDqk = 576;     // 512 latent + 64 RoPE dims
constexpr int kDv = 512;      // value = first 512 dims of the latent row
constexpr int kPage = 64;     // tokens per page = tokens per tile
constexpr int kChunk = 64;    // dims per 128-byte swizzle atom row (bf16)
constexpr int kNumChunks = kDqk / kChunk;  // 9
// CTA 0 of a pair owns dims [0, 256) (score part and O columns); CTA 1 owns
// dims [256, 576) for the score and O columns [256, 512).
constexpr int kSplitDim = 256;
constexpr int kVcolsPerCta = kDv / 2;  // 256

// Workspace layout (all offsets in bytes, 256-aligned sections).
struct WsLayout {
  size_t hdr, units, reqs, part_lse, part_o, total;
  int slots;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

__host__ __device__ inline WsLayout ws_layout(int batch, int s_q, int num_units) {
  WsLayout L;
  L.slots = 2 * num_units;  // a plan never needs more than 2 * (units - 1)
  size_t off = 0;
  L.hdr = off;      off += align256(64 * sizeof(int));
  L.units = off;    off += align256(static_cast<size_t>(num_units) * 5 * sizeof(int));
  L.reqs = off;     off += align256(static_cast<size_t>(batch) * 4 * sizeof(int));
  L.part_lse = off; off += align256(static_cast<size_t>(L.slots) * s_q * kHeads * sizeof(float));
  L.part_o = off;   off += align256(static_cast<size_t>(L.slots) * s_q * kHeads * kDv * sizeof(uint16_t));
  L.total = off;
  return L;
}

// Header words of the workspace.
enum { kHdrStatus = 0, kHdrUnits = 1, kHdrWidth = 2, kHdrTotal = 3, kHdrSlots = 4 };

// Device status codes (same numbering as the public mla_status).
enum { kStOk = 0, kStWorkspace = 3, kStBadTable = 6, kStBadIndex = 7, kStTimeout = 8, kStValueRange = 9 };

// Host-side argument checks of mla_decode (status code; MLA_OK = 0).
int check_decode_args(const void* q, const void* kv_cache, int64_t num_pages, const int32_t* block_table,
                      int64_t bt_stride, const int32_t* cache_lens, int batch, int s_q, int num_heads,
                      float softmax_scale, const int32_t* topk_idx, int topk, unsigned flags, const void* out,
                      const float* lse);

struct DecodeParams {
  const uint16_t* q;          // bf16 [B, s_q, 128, 576]
  const uint16_t* kv;         // bf16 [num_pages, 64, 576]
  const int* block_table;     // [B, bt_stride]
  long long bt_stride;
  const int* cache_lens;      // [B]
  const int* topk_idx;        // [B, s_q, topk] or null
  int topk;
  int batch;
  int s_q;
  int causal;
  long long num_pages;
  float scale_log2;           // softmax_scale * log2(e)
  void* out;                  // bf16 or fp32 [B, s_q, 128, 512]
  float* lse;                 // [B, s_q, 128]
  int out_fp32;
  int num_units;
  int* ws_hdr;
  const int* unit_meta;       // [U, 5]
  const int* req_meta;        // [B, 4]
  float* part_lse;            // [slots, s_q, 128]
  uint16_t* part_o;           // [slots, s_q, 128, 512], fp16 (bf16 when part_bf16)
  int part_bf16;              // partial rows in bf16 (MLA_FLAG_BF16_PV) instead of fp16
};

}  // namespace mla
