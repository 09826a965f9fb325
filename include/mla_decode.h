/*
 * mla_decode.h — C ABI of the GB300 (sm_103a) MLA decode library.
 *
 * The operation
 * -------------
 * Weight-absorbed multi-head latent attention at decode time ("DeepSeek
 * V3/R1 Inference Efficiency (2): Reverse-Engineering the Production
 * Deployment", §2.4.1, Compute, "MLA/MQA attention"): each of a request's
 * 128 query heads carries 576 dims (512 latent + 64 RoPE) and attends, in MQA
 * form, over the request's cached latent rows (576 bf16 per token).  The
 * score contraction spans all 576 dims, the value is the first 512 dims of
 * the same row.  For request b, query token t and head h:
 *
 *     s_j = scale * <q[b,t,h,:], kv[row(j),:]>          j visible
 *     O[b,t,h,:] = sum_j softmax(s)_j * kv[row(j), 0:512]
 *     LSE[b,t,h] = ln sum_j exp(s_j)                      (natural log)
 *
 * The cache lives in 64-token pages of a shared pool reached through a block
 * table ("How DeepSeek Inference Works", levers table, "KV-cache layout (MLA,
 * paging)"): logical position j of request b is pool row
 * block_table[b * bt_stride + j / 64] * 64 + j % 64.
 *
 * Long or skewed lengths are split across the GPU (split-KV, the split-K
 * remedy of "The 31-Millisecond Smoking Gun" and the wave-quantisation
 * discussion of "The Premise That Wasn't", Wave-Aware NSPLIT); partial
 * results are merged with LSE weights.
 *
 * Three calls make one decode step, all asynchronous on `stream`:
 *     mla_decode_plan  -> partitions the (request, 64-token tile) work
 *     mla_decode       -> attention; writes final O/LSE for unsplit requests
 *                         and 16-bit partials (fp16; bf16 with
 *                         MLA_FLAG_BF16_PV) plus fp32 LSEs for split ones
 *     mla_combine      -> merges the partials, writes O/LSE of split requests
 *                         and of requests with nothing to attend to
 *
 * Conventions
 * -----------
 *  - Every pointer is a DEVICE pointer unless stated otherwise.  The caller
 *    owns all memory; the library allocates nothing.
 *  - The return value reports errors detectable on the host (bad arguments,
 *    unsupported shapes or device, launch failures).  Errors found on the
 *    device (validate mode, a wait that ran out) are recorded in the
 *    workspace's status word; the kernels of the step that find it set leave
 *    their outputs unwritten, and mla_workspace_status (mla_noalloc_status
 *    for the built-in workspace) reports it.  Only those two status queries
 *    synchronise the stream; every other call is asynchronous and can be
 *    recorded into a CUDA graph.
 *  - Fixed shapes: 128 query heads, 576 q/k dims, 512 value dims, 64-token
 *    pages.  Anything else returns MLA_ERR_UNSUPPORTED.  The device must be
 *    compute capability 10.3 (GB300); there is no other code path.
 *  - The plan lives in the caller's workspace; the three calls of one step
 *    must use the same workspace, batch, s_q, topk and num_units.
 *  - Calls are stateless and thread-safe for distinct workspaces.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream (cudaStream_t); NULL means the legacy default stream. */
typedef void* mla_stream_t;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,  /* null pointer, negative size, misalignment   */
  MLA_ERR_UNSUPPORTED = 2,  /* head count / dims / device not supported     */
  MLA_ERR_WORKSPACE = 3,    /* workspace too small                          */
  MLA_ERR_CUDA = 4,         /* a CUDA runtime or driver call failed         */
  MLA_ERR_DEVICE = 5,       /* no sm_103 device current                     */
  MLA_ERR_BAD_TABLE = 6,    /* validate mode: block-table entry / length out of range */
  MLA_ERR_BAD_INDEX = 7,    /* validate mode: top-k index outside [-1, len) */
  MLA_ERR_TIMEOUT = 8,      /* a device-side wait ran out (kernel bailed out) */
  MLA_ERR_VALUE_RANGE = 9   /* validate mode: a value dim the step reads is not
                               finite or does not fit fp16 (|v| >= 65536) */
} mla_status;

enum {
  MLA_FLAG_CAUSAL = 1,   /* s_q >= 2 (MTP decode): token t sees [0, len - s_q + t] */
  MLA_FLAG_OUT_FP32 = 2, /* O is written as fp32 instead of bf16           */
  MLA_FLAG_VALIDATE = 4, /* check lengths, table, indices and value range
                            first; see mla_decode                           */
  MLA_FLAG_BF16_PV = 8   /* s_q = 2 dense only: the value product takes the
                            softmax weights and values in bf16 (8 significant
                            bits on the weights) instead of the default fp16
                            (11 bits).  No value-range limit, but on a peaked
                            softmax (a few rows of large magnitude dominating)
                            the O error grows to a few times 2e-2.  Every
                            other path, and this one by default, computes the
                            value product in fp16: value dims must then stay
                            below 65504 in magnitude.  On every path the flag
                            also stores split requests' partial rows in bf16
                            instead of fp16 (as wide in range as the values) */,
  MLA_FLAG_KV_FP8 = 16   /* the cache is FP8 (see MLA_FP8_ROW_BYTES): the
                            latent caching in FP8 of "The 31-Millisecond
                            Smoking Gun" (DeepSeek-V4-Flash paragraph) and the
                            precision lever of "How DeepSeek Inference Works".
                            Every s_q, dense or top-k; all run the one-token
                            kernel (for s_q = 2 dense, one 2-CTA cluster per
                            token on the plan's two-page tiles, in place of
                            the paired-SM kernel, which has no FP8 form).
                            mla_combine accepts the flag and ignores it. */
};

/*
 * FP8 cache rows (MLA_FLAG_KV_FP8).  The pages give no byte format; the
 * reading implemented is a 656-byte row per cached token:
 *   bytes [0, 512)    the 512 latent dims as OCP FP8 E4M3 codes (bias 7, no
 *                     infinities, S.1111.111 = NaN)
 *   bytes [512, 516)  one UE8M0 scale per 128-dim group of the latent:
 *                     scale = 2^(byte - 127)
 *   bytes [516, 528)  unused
 *   bytes [528, 656)  the 64 RoPE dims in bf16
 * Latent dim d = e4m3(byte d) * scale[d / 128].  With an FP8 cache both
 * products take the latent dims in fp16 (the query's too; the RoPE dims stay
 * bf16): power-of-two scales make every cached value exact in fp16 within
 * its range, so the step attends over exactly the values the rows encode,
 * provided the cached values and the query's latent dims stay below 65504 in
 * magnitude (query dims below 2^-14 round to fp16 subnormals).  A page is 64
 * rows (41,984 bytes); the block table is unchanged.
 */
enum { MLA_FP8_ROW_BYTES = 656 };

enum { MLA_NUM_HEADS = 128, MLA_D_QK = 576, MLA_D_V = 512, MLA_PAGE = 64, MLA_MAX_SQ = 8 };

/*
 * Number of persistent work units that `num_units = 0` selects on the
 * current device.  s_q = 1: one unit is a pair of SMs working as a 2-CTA
 * cluster, and the count is the number of co-resident 2-CTA clusters.
 * s_q = 2: a dense unit is a 4-CTA cluster (two SM pairs) serving both query
 * tokens, a top-k unit is two 2-CTA clusters (one per token); the count is
 * what both forms keep resident.  s_q = 3 .. MLA_MAX_SQ: a unit is s_q 2-CTA
 * clusters, one per token (each token's cluster reads the request's pages;
 * the repeats are served by L2).  Host-only; returns 0 and sets *err on
 * failure (err may be NULL).
 */
int mla_default_num_units(int s_q, int* err);

/*
 * Bytes of workspace the three calls need.  Pure host arithmetic.
 *   batch      requests (>= 1)
 *   s_q        query tokens per request (1 .. MLA_MAX_SQ)
 *   num_heads  must be 128
 *   num_units  work units per query token; 0 = mla_default_num_units(s_q)
 * Returns 0 on invalid arguments.
 */
size_t mla_decode_workspace_size(int batch, int s_q, int num_heads, int num_units);

/*
 * Split-KV partition of one decode step.  Launches one CTA; reads
 * cache_lens on the device, so no host synchronisation is needed.
 *   cache_lens  int32 [batch], tokens in each request's cache (>= 0)
 *   topk        0 for dense attention; else the length of each top-k list
 *               (every request then has ceil(topk / 64) tiles)
 *   num_units   as for mla_decode_workspace_size
 *   workspace   device buffer of ws_bytes >= mla_decode_workspace_size(...)
 * The work of request b is ceil(len_b / R) tiles of R tokens (R = 128 for
 * s_q = 2 dense, whose kernel takes two pages per step; else 64); the tiles
 * of all requests, each request charged a fixed per-split overhead, are cut
 * into num_units contiguous, equally loaded ranges.  Requests that straddle
 * a cut are "split" and finish in mla_combine.
 */
int mla_decode_plan(const int32_t* cache_lens, int batch, int s_q, int topk,
                    int num_units, void* workspace, size_t ws_bytes,
                    mla_stream_t stream);

/*
 * The same partition computed on the host from host-resident lengths, for
 * inspection and testing.  Writes, per unit u, unit_meta[5u .. 5u+4] =
 * {begin_req, begin_tile, end_req, end_tile, first_split} (ranges are
 * half-open in (request, tile) order), and per request b,
 * req_meta[4b .. 4b+3] = {n_tiles, n_splits, first_slot, cost_prefix}.
 * unit_meta holds 5 * num_units ints and req_meta 4 * batch ints (host
 * memory, caller-owned).  num_units must be >= 1 here.
 */
int mla_decode_plan_host(const int32_t* cache_lens_host, int batch, int s_q,
                         int topk, int num_units, int32_t* unit_meta,
                         int32_t* req_meta);

/*
 * Attention for one decode step (after mla_decode_plan on the same stream).
 *   q            bf16 [batch, s_q, 128, 576], contiguous, 16-B aligned
 *   kv_cache     bf16 [num_pages, 64, 576], contiguous, 16-B aligned; with
 *                MLA_FLAG_KV_FP8 bytes [num_pages, 64, 656] (FP8 rows)
 *   num_pages    pages in the pool (rows = 64 * num_pages)
 *   block_table  int32, row b at block_table + b * bt_stride; entries
 *                0 .. ceil(len_b / 64) - 1 are read
 *   bt_stride    elements between block-table rows (>= ceil(max len / 64))
 *   cache_lens   int32 [batch]
 *   s_q          1 .. MLA_MAX_SQ (with MLA_FLAG_CAUSAL for MTP decode:
 *                the request's last s_q cached tokens are its query tokens)
 *   num_heads    must be 128
 *   softmax_scale  multiplies the 576-dim dot product (used as float32)
 *   topk_idx     NULL for dense attention; else int32 [batch, s_q, topk] of
 *                logical positions in the request's sequence, -1 = unused
 *                slot; each list attends to exactly its entries (CAUSAL is
 *                then ignored)
 *   flags        MLA_FLAG_*
 *   workspace    the planned workspace
 *   out          [batch, s_q, 128, 512], bf16 (or fp32 with OUT_FP32)
 *   lse          fp32 [batch, s_q, 128], natural log; -inf where nothing
 *                is visible (O is then 0)
 * Out-of-range table entries or indices never fault: dense page loads
 * outside the pool read zeros, sparse rows outside it are skipped; results
 * for such requests are meaningless.  MLA_FLAG_VALIDATE detects them first:
 * a check kernel runs before the attention on the same stream and records
 * MLA_ERR_BAD_TABLE, MLA_ERR_BAD_INDEX or (wherever the value product is
 * fp16, i.e. everywhere but the MLA_FLAG_BF16_PV two-token path)
 * MLA_ERR_VALUE_RANGE for a visible value dim that is not finite or has
 * |v| >= 65536 (FP8 rows: a NaN code, a scale byte of 255, or a scaled
 * latent dim of 65536 or more); the attention and combine kernels then leave O and LSE
 * unwritten.  It reads every visible cache row once more (a full pass over
 * the cache: a debugging aid, not a production mode).  The call does not
 * synchronise: read the outcome with mla_workspace_status.
 * A device-side wait that runs out (about 2 s) makes the kernel record
 * MLA_ERR_TIMEOUT in the workspace and return; mla_workspace_status reads it.
 */
int mla_decode(const void* q, const void* kv_cache, int64_t num_pages,
               const int32_t* block_table, int64_t bt_stride,
               const int32_t* cache_lens, int batch, int s_q, int num_heads,
               float softmax_scale, const int32_t* topk_idx, int topk,
               unsigned flags, int num_units, void* workspace, size_t ws_bytes,
               void* out, float* lse, mla_stream_t stream);

/*
 * Merge the split requests' partials (LSE = ln sum_s exp(lse_s),
 * O = sum_s exp(lse_s - LSE) * O_s) and write O = 0, LSE = -inf for
 * requests with nothing to attend to.  flags: MLA_FLAG_OUT_FP32 as above,
 * and MLA_FLAG_BF16_PV as given to mla_decode (it sets the partials' format).
 */
int mla_combine(void* workspace, size_t ws_bytes, int batch, int s_q,
                int num_heads, unsigned flags, int num_units, void* out,
                float* lse, mla_stream_t stream);

/*
 * Synchronise `stream` and return the device-side status recorded in the
 * workspace: MLA_OK; MLA_ERR_BAD_TABLE, MLA_ERR_BAD_INDEX or
 * MLA_ERR_VALUE_RANGE from validate mode; MLA_ERR_TIMEOUT; or a plan
 * overflow as MLA_ERR_WORKSPACE.  mla_decode_plan resets it to MLA_OK.
 */
int mla_workspace_status(const void* workspace, mla_stream_t stream);

/*
 * The same decode step (plan + attention + combine) for callers that cannot
 * allocate device memory when it runs: a runtime that records its per-token
 * work into a CUDA graph (allocation is not allowed during stream capture),
 * or a host program with a fixed device-memory budget that forbids any
 * allocation after start-up.  There is no counterpart of this call in the
 * method's description; it only changes where the workspace lives.
 *
 * Arguments are those of mla_decode, without workspace and num_units.  The
 * workspace is a 48 MiB array inside the library's device image, which every
 * GPU that loads the library keeps until the process exits.  The number of
 * work units is mla_default_num_units(s_q), lowered if the workspace of
 * (batch, s_q) would not fit; MLA_ERR_WORKSPACE if it does not fit even with
 * one unit.  The call allocates nothing.  Its first call on a device looks up
 * the array's device address (with that device current); make that first
 * call before any stream capture.  All calls share the array: calls whose
 * work overlaps on the GPU (other streams, other host threads) race and must
 * be serialised by the caller.  Errors found on the device (validate mode, a
 * wait that ran out) are read with mla_noalloc_status.
 */
int mla_decode_noalloc(const void* q, const void* kv_cache, int64_t num_pages,
                       const int32_t* block_table, int64_t bt_stride,
                       const int32_t* cache_lens, int batch, int s_q, int num_heads,
                       float softmax_scale, const int32_t* topk_idx, int topk,
                       unsigned flags, void* out, float* lse, mla_stream_t stream);

/*
 * Synchronise `stream` and return the status word of the built-in workspace
 * of mla_decode_noalloc on the current device: the codes of
 * mla_workspace_status (a failed validation, a wait that ran out).  Each
 * mla_decode_noalloc call resets it when its plan runs.
 */
int mla_noalloc_status(mla_stream_t stream);

/*
 * Device address and size in bytes of the built-in workspace on the current
 * device (looked up on first use, like mla_decode_noalloc), for diagnostics
 * such as mla_selftest_wait_timeout.  Returns MLA_ERR_INVALID_ARG for null
 * pointers.
 */
int mla_noalloc_workspace(void** dev_ptr, size_t* bytes);

/*
 * Diagnostic of the device-side failure path (no counterpart in the method's
 * description).  Launches one CTA on `stream` that waits, with the bounded
 * wait every decode kernel uses, on a shared-memory barrier that nothing
 * completes.  The wait gives up after its limit (about 2 s), records
 * MLA_ERR_TIMEOUT in the workspace header (the word mla_workspace_status
 * reads) and the kernel returns: no trap, no fault, the context stays usable.
 * `workspace` is a decode workspace of at least 256 bytes (device pointer,
 * 256-byte aligned); only its status word is written.  Returns MLA_OK once
 * launched (asynchronous), MLA_ERR_INVALID_ARG for a bad workspace, or a
 * launch error.
 */
int mla_selftest_wait_timeout(void* workspace, size_t ws_bytes, mla_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* mla_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
