// decode_kernel.cu — weight-absorbed MLA decode attention on sm_103a.
//
// What it computes ("DeepSeek V3/R1 Inference Efficiency (2)", §2.4.1,
// Compute, "MLA/MQA attention"): every request's 128 query heads (576 dims:
// 512 latent + 64 RoPE) attend over the request's cached latent rows; scores
// contract all 576 dims, values are the first 512 dims of the same row.
// Cached rows sit in 64-token pages reached through a block table.
//
// One work unit = one 2-CTA cluster on a pair of SMs.  The fp32 output
// O = 128 heads x 512 fills one SM's whole tensor memory, so the pair splits
// the work by stage of the attention rather than by dimension:
//
//   CTA 0, "S side": Q (128 x 576 bf16) lives in tensor memory as the A
//     operand; per 64-token tile it computes S = Q K^T on tcgen05 (M=128,
//     N=64, K=576, fp32 in TMEM), runs the online softmax in fp32 (exp2
//     domain, lazy rescale: the reference max moves only when a score beats
//     it by more than 2^8) and streams the fp16 weights P plus a per-row
//     rescale factor into CTA 1's shared memory with st.async, which
//     completes on CTA 1's mbarrier (no round trip, no fence).
//   CTA 1, "O side": owns O (128 x 512 fp32, all 512 TMEM columns); per tile
//     it converts the value part of the tile to fp16 in shared memory (values
//     must stay below 65504 in magnitude), rescales O rows when the
//     S side moved the max, and accumulates O += P V on tcgen05 (M=128,
//     N=2x256, K=64).  P and V in fp16 keep 11 significant bits on the
//     softmax weights (bf16 would keep 8), which is what holds the O error
//     under 2e-2 when a few rows dominate the softmax.
//
// Both CTAs fetch the tile with TMA (the O side only the 512 value dims);
// the second fetch of the pair is served by L2.  A persistent grid walks the
// split-KV plan: a request cut by a unit boundary writes a normalised fp32
// partial plus its LSE, merged by the combine kernel (the split-K remedy of
// "The 31-Millisecond Smoking Gun").
//
// Warps (384 threads dense, 640 top-k).  S side: 0-7 softmax (warp w: head
// rows 32*(w%4).., columns 32*(w/4).. of each tile), 8 MMA issue + TMEM
// owner, 9 TMA producer (dense) or, with 10-19, row gather (top-k).  O side:
// 0-3 O correction + epilogue (thread i = head row i = TMEM lane i), 4-7 and
// 10-11 V conversion (dense) or 4-7 and 10-19 row gather + conversion
// (top-k), 8 MMA issue, 9 TMA producer (dense).  (The gather is issue-bound:
// 20 warps measured 6 % faster than 16 on the top-2048 workload.)
//
// FP8 latent cache (kFp8, MLA_FLAG_KV_FP8; 640 threads): a cached token is a
// 656-byte row of 512 E4M3 latent dims, four UE8M0 (power-of-two) scales,
// one per 128-dim group, and the 64 RoPE dims in bf16.  A tile's latent and
// scale bytes (64 rows x 528 B) land at the end of the stage's eight latent
// chunks (TMA, or the top-k row gather) and fill warps widen them in place:
// every fill thread first reads its share of the raw bytes into registers,
// the group meets at a named barrier, then each thread writes its pieces as
// fp16 in the 128B-swizzled chunk layout: one convert and one multiply by
// the power-of-two scale per two codes.  Both products then run in fp16 over
// the latent dims: the S side also widens Q's 512 latent dims to fp16 (once
// per segment, in its ring slots); the RoPE dims stay bf16 in both operands
// (the score MMAs of chunk 8 take the bf16 descriptor).  A code times its
// scale is exact in fp16 within its range (values and query latent dims below
// 65504 in magnitude), so the attention reads exactly the cached values.  Fill
// warps: S side 10-19 (dense, warp 9 issues the TMA loads) or 9-19 (top-k),
// O side 4-7 and 10-19; the MMA thread waits for the fill threads' arrivals
// (kVR) on every ring slot, Q slots included.  (The fill work is latency-
// bound: 20 warps, so that 10-14 of them fill, measured faster than 16.)
// Two query tokens over a dense FP8 cache (which the paired-SM two-token
// kernel does not read) run here too, one cluster per token, on the plan
// the paired-SM kernel would get: the kPairTiles instance splits each of its
// 128-row tiles into two of this kernel's 64-row tiles (Seg64Iter).
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernel_common.cuh"
#include "plan.cuh"
#include "ptx.cuh"

namespace mla {

// 32-byte global store (one whole L2 sector); the address must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               ::"l"(p), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

constexpr int kChunkBytes = kPage * 128;         // 64 rows x 64 bf16, 128B-swizzled
constexpr int kStages = 3;
constexpr int kStageS = kNumChunks * kChunkBytes;  // 9 chunks: all 576 dims
constexpr int kStageO = 8 * kChunkBytes;           // 8 chunks: the 512 value dims
constexpr int kPBytes = kHeads * 128;              // 128 rows x 64 fp16
constexpr int kQChunkBytes = kHeads * 128;         // Q: 128 rows x 64 bf16, 128B-swizzled

// FP8 latent cache: a row's latent + scale bytes (528 of 656) land at the
// end of the eight latent chunks of a stage and are widened there.
constexpr int kF8Row = 656;                                // bytes per cached token
constexpr int kF8Lat = 528;                                // 512 E4M3 codes, 4 scale bytes, 12 unused
constexpr int kF8RawBytes = kF8Lat * kPage;                // 33,792 per tile
constexpr int kF8RawOff = 8 * kChunkBytes - kF8RawBytes;   // 31,744
constexpr int kF8Pieces = 8 * kPage * 4;                   // 16-byte raw pieces (16 codes) per tile
constexpr int kF8Low = 3 * kPage * 4;                      // pieces of chunks 0-2: outputs below the raw bytes
constexpr int kF8PerThread = (kF8Pieces - kF8Low + 319) / 320;  // 4: buffered pieces of chunks 3-7 per thread
static_assert(kF8RawOff % 16 == 0, "TMA destination alignment");
// FP8 kernels run 20 warps; fill threads: S side warps 10-19 (dense) or 9-19
// (top-k); O side 4-7 and 10-19
constexpr int kThreadsFp8 = 640;
__host__ __device__ constexpr int f8_fill_threads(bool sparse, bool s_side) {
  return s_side ? (sparse ? 352 : 320) : 448;
}

// Shared-memory layout (offsets from a 1024-aligned base).  The barrier block
// sits at the same offset in both CTAs (multicast commits rely on it).
constexpr int kOffStage = 0;
constexpr int kOffP = kStages * kStageO;             // O side: 196608
constexpr int kOffAlpha = kOffP + 2 * kPBytes;       // O side: float[2][128]
constexpr int kOffFin = kOffAlpha + 2 * kHeads * 4;  // O side: float[2][128]
constexpr int kOffBar = kOffFin + 2 * kHeads * 4;    // 231424
constexpr int kOffXchg = kStages * kStageS;          // S side: row max / sum exchange, 4 KiB
constexpr int kBarBytes = 256;
constexpr int kSmemUsed = kOffBar + kBarBytes;
constexpr int kAlignSlack = 768;
constexpr int kSmemBytes = kSmemUsed + kAlignSlack;  // 232448 = the opt-in maximum
static_assert(kOffXchg + 4096 <= kOffBar, "S-side stages overlap the barrier block");

// Tensor-memory columns.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;     // S side: two 64-column score buffers
constexpr uint32_t kColQ = 128;   // S side: Q, 288 columns (576 bf16 packed in pairs)
constexpr uint32_t kColO = 0;     // O side: O, 512 columns

constexpr int kThreads = 384;       // 12 warps (dense); the top-k variant has 16
constexpr int kThreadsSparse = 640;
// O side: warps 4-7 and 10-11 convert V (dense); warps 4-7 and 10-19 gather
// and convert it (top-k)
__host__ __device__ constexpr int conv_threads(bool sparse) { return sparse ? 448 : 192; }
constexpr float kRescaleLog2 = 8.0f;

enum Bar {
  kKF = 0,        // [3] tile landed (TMA tx, or 128 gather arrivals)
  kKE = 3,        // [3] tile free (MMA commit)
  kVR = 6,        // [3] O side: fp16 V ready (128 arrivals)
  kQR = 9,        // (unused)
  kQF = 10,       // S side: Q free (commit after a segment's last QK)
  kSF = 11,       // [2] S side: scores ready (commit)
  kSE = 13,       // [2] S side: scores read (128 arrivals)
  kPFree = 15,    // [2] S side: O side finished PV on that P slot (remote commit)
  kPM = 17,       // [2] O side: P message landed (1 arrival + tx bytes)
  kPR = 19,       // [2] O side: O corrected, PV may go (128 arrivals)
  kPD = 21,       // [2] O side: PV of a tile of that parity finished (commit)
  kOF = 23,       // O side: segment's last PV finished (commit)
  kOE = 24,       // O side: epilogue read O (128 arrivals)
  kMmaDone = 25,  // teardown
  kNumBars = 26
};
static_assert(kNumBars * 8 + 16 <= kBarBytes, "barrier block");

// kind::f16 instruction descriptors: S = Q K^T with bf16 operands; O += P V
// with fp16 operands (A and B of one MMA always share a type).
constexpr uint32_t kIdescQK = idesc_bf16(128, 64, 0);
// FP8 cache: the scores take Q and K in fp16 (A and B formats 0) over the
// 512 latent dims, in bf16 over the 64 RoPE dims (chunk 8)
constexpr uint32_t kIdescQK16 = kIdescQK & ~((1u << 7) | (1u << 10));
constexpr uint32_t kIdescPV = (1u << 4) | (0u << 7) | (0u << 10) | (1u << 16) | ((256u >> 3) << 17) |
                              ((128u >> 4) << 24);

// The segments of a unit in this kernel's 64-row tiles.  A plan made for
// two query tokens over a dense cache counts 128-row tiles (kPairTiles: the
// tiles of the paired-SM kernel, which an FP8 cache does not use): each
// becomes two, and a segment that ends its request stops at the request's
// last page.
template <bool kPairTiles>
struct Seg64Iter {
  SegIter it;
  const int* lens;
  __device__ Seg64Iter(const DecodeParams& p, int unit) : it(p, unit), lens(p.cache_lens) {}
  __device__ bool next(Seg& s) {
    while (it.next(s)) {
      if (kPairTiles) {
        const bool to_end = s.t1 == s.n_tiles;
        s.t0 *= 2;
        s.t1 *= 2;
        if (to_end) {
          const int n64 = (max(lens[s.b], 0) + kPage - 1) / kPage;
          s.t1 = min(s.t1, n64);
        }
        if (s.t0 >= s.t1) continue;
      }
      return true;
    }
    return false;
  }
};

// Position in the 3-deep tile ring.
struct Ring3 {
  uint32_t idx = 0, phase = 0;
  __device__ void advance() {
    if (++idx == kStages) { idx = 0; phase ^= 1u; }
  }
};

// tcgen05.mma with the A operand in tensor memory.
__device__ __forceinline__ void umma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Two E4M3 codes (bits 0-7: the lower dim) -> fp16x2 (exact: every E4M3
// value is an fp16 normal or zero).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t r;
  asm("{\n .reg .b16 c;\n cvt.u16.u32 c, %1;\n cvt.rn.f16x2.e4m3x2 %0, c;\n}" : "=r"(r) : "r"(two_codes));
  return r;
}

// fp16x2 times a power-of-two scale -> bf16x2 (S side) or fp16x2 (O side).
template <bool kToBf16>
__device__ __forceinline__ uint32_t scale_f16x2(uint32_t h2, float s) {
  float lo, hi;
  asm("{\n .reg .f16 a, b;\n mov.b32 {a, b}, %2;\n cvt.f32.f16 %0, a;\n cvt.f32.f16 %1, b;\n}"
      : "=f"(lo), "=f"(hi) : "r"(h2));
  return kToBf16 ? pack_bf16x2(lo * s, hi * s) : pack_f16x2(lo * s, hi * s);
}

// The scale 2^(E - 127) of a UE8M0 byte as two fp16x2 multipliers m1 * m2:
// m1 = 2^clamp(E - 127, -24, 15) (an fp16 power of two, subnormal below
// 2^-14), m2 the rest (1 for E in [103, 142]; else a power of two that
// underflows to 0 or overflows to infinity as fp16 would).
__device__ __forceinline__ uint2 f16_scale_pair(uint32_t E) {
  const int k = static_cast<int>(E) - 127;
  const int k1 = k < -24 ? -24 : (k > 15 ? 15 : k);
  const int k2 = k - k1;
  auto pow2 = [](int e) -> uint32_t {  // 2^e as fp16 bits
    if (e > 15) return 0x7c00u;
    if (e >= -14) return static_cast<uint32_t>(e + 15) << 10;
    if (e >= -24) return 1u << (e + 24);
    return 0u;
  };
  const uint32_t m1 = pow2(k1), m2 = pow2(k2);
  return make_uint2(m1 | (m1 << 16), m2 | (m2 << 16));
}

// 16 E4M3 codes (a raw piece, dims in byte order) times the scale (m) -> 8
// fp16x2 words: one convert and one multiply (two outside [103, 142]) per two
// codes.  Exact wherever the result is an fp16 (normal, or subnormal on its
// 2^-24 grid), which covers |v| in [2^-14, 65504].  (Placing the code bits
// with integer operations instead measured slower, also with 20 warps.)
__device__ __forceinline__ void widen_f16(uint4 v, uint2 m, uint32_t (&w)[8]) {
  const uint32_t in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t a, b;
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n cvt.rn.f16x2.e4m3x2 %1, hi;\n}"
        : "=r"(a), "=r"(b) : "r"(in[i]));
    asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(a) : "r"(m.x));
    asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(b) : "r"(m.x));
    if (m.y != 0x3c003c00u) {
      asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(a) : "r"(m.y));
      asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(b) : "r"(m.y));
    }
    w[2 * i] = a;
    w[2 * i + 1] = b;
  }
}

// In place: the 16-byte pieces piece0, piece0 + step, ... (< n) of the bf16
// region at `base` -> fp16 (exact within fp16's range).
__device__ __forceinline__ void bf16_region_to_f16(uint32_t base, int piece0, int step, int n) {
  for (int i = piece0; i < n; i += step) {
    const uint32_t a = base + 16u * static_cast<uint32_t>(i);
    const uint4 v = ld_shared_v4u(a);
    st_shared_v4(a, bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
  }
}

// UE8M0 byte -> 2^(byte - 127) as fp32 (byte 0 is the subnormal 2^-127).
__device__ __forceinline__ float ue8m0_scale(uint32_t byte) {
  return byte ? __uint_as_float(byte << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ uint32_t ld_shared_u8(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}

// Commit that arrives on the mbarrier at the same offset in every CTA of `mask`.
__device__ __forceinline__ void umma_commit_multicast(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar), "h"(mask) : "memory");
}

// Bytes of one P message (fp16 P tile, per-row rescale, and at the end of a
// segment the per-row final scale).
__host__ __device__ constexpr uint32_t p_message_bytes(bool last) {
  return static_cast<uint32_t>(kPBytes + kHeads * 4 + (last ? kHeads * 4 : 0));
}

template <bool kSparse, bool kFp8, bool kPairTiles = false>
__global__ void __launch_bounds__(kFp8 ? kThreadsFp8 : (kSparse ? kThreadsSparse : kThreads), 1)
mla_decode_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_rope) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t mis = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + mis;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int U = p.num_units;
  const int cluster_id = blockIdx.x >> 1;
  const int unit = cluster_id % U;
  const int tok = cluster_id / U;
  const bool s_side = rank == 0;
  grid_launch_dependents();  // the combine kernel may be scheduled now; it waits for this grid
  grid_dependency_wait();    // the plan of this step is complete (programmatic dependent launch)

  {  // a unit with no work leaves at once (both CTAs see the same range), and
     // so does every unit once the step's status word is set (a failed
     // validation): the plan and the check are complete here, and nothing
     // else writes the word before this grid's own waits could run out
    const int* um = p.unit_meta + 5 * unit;
    if (um[0] >= p.batch || (um[0] == um[2] && um[1] >= um[3])) return;
    if (p.ws_hdr[kHdrStatus] != 0) return;
  }
  if (mis > kAlignSlack) {  // never touch shared memory past the end of the allocation
    if (threadIdx.x == 0) atomicCAS(p.ws_hdr + kHdrStatus, 0, static_cast<int>(kStWorkspace));
    return;
  }

  const uint32_t sStage = sbase + kOffStage;
  const uint32_t sP = sbase + kOffP;
  const uint32_t sAlpha = sbase + kOffAlpha;
  const uint32_t sFin = sbase + kOffFin;
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * static_cast<uint32_t>(i); };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * kNumBars);
  // misc[0] = TMEM base address, misc[1] = abort flag
  const int stage_bytes = s_side ? kStageS : kStageO;
  const int nchunks = s_side ? kNumChunks : 8;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kKF + i), 1);
      mbar_init(bar(kKE + i), 1);
      mbar_init(bar(kVR + i), kFp8 ? f8_fill_threads(kSparse, s_side) : conv_threads(kSparse));
    }
    mbar_init(bar(kQF), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kSF + i), 1);
      mbar_init(bar(kSE + i), 256);
      mbar_init(bar(kPFree + i), 1);
      mbar_init(bar(kPM + i), 1);
      mbar_init(bar(kPR + i), 128);
    }
    mbar_init(bar(kPD), 1);
    mbar_init(bar(kPD + 1), 1);
    mbar_init(bar(kOF), 1);
    mbar_init(bar(kOE), 128);
    mbar_init(bar(kMmaDone), 1);
    misc[1] = 0u;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(smem_u32(&misc[0]), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 9 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kv);
    tma_prefetch_desc(&tm_rope);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before any remote operation
  tc_fence_after();
  const uint32_t tmem = misc[0];

  Ctl ctl;
  ctl.abort = &misc[1];
  ctl.abort_remote[0] = mapa(smem_u32(&misc[1]), peer);
  ctl.n_remote = 1;
  ctl.status = p.ws_hdr + kHdrStatus;
  const float NEG_INF = -__int_as_float(0x7f800000);

  if (warp < 8 && s_side) {
    // ================================================= S side: Q load + softmax
    // Warp w handles head rows 32*(w%4) .. +31 (its TMEM lane quarter) and
    // columns 32*(w/4) .. +31 of every 64-token tile; the two warps of a
    // quarter swap their partial row max through shared memory.
    const int q4 = warp & 3, half = warp >> 2;
    const int row = q4 * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t rP = mapa(sP, peer) + static_cast<uint32_t>(row) * 128u;
    const uint32_t rAlpha = mapa(sAlpha, peer) + static_cast<uint32_t>(row) * 4u;
    const uint32_t rFin = mapa(sFin, peer) + static_cast<uint32_t>(row) * 4u;
    const uint32_t rPM = mapa(bar(kPM), peer);
    float* xmax = reinterpret_cast<float*>(smem + kOffXchg);               // [2 parity][2 half][128]
    float* xsum = reinterpret_cast<float*>(smem + kOffXchg + 4 * kHeads * 4);  // [2 half][2][128]
    const int pair_bar = 1 + q4;  // named barrier of the two warps of this quarter
    // the two warps of a quarter meet at named barriers: they vote there, so
    // that a wait that ran out in one of them makes both leave
    Seg64Iter<kPairTiles> it(p, unit);
    Seg sg;
    uint32_t g = 0, nseg = 0;
    bool ok = true, stop = false;  // ok: this warp's waits so far; stop: the quarter leaves
    while (!stop && it.next(sg)) {
      const int L = max(p.cache_lens[sg.b], 0);
      const int vis = p.causal ? L - p.s_q + tok + 1 : L;
      const long long bt_row = static_cast<long long>(sg.b) * p.s_q + tok;
      // z: sum of the fp16-rounded weights (normalises O, whose PV product uses
      // exactly those weights); zx: sum of the unrounded weights (for the LSE).
      // Each half keeps the sums of its own columns.
      float m_used = NEG_INF, z = 0.f, zx = 0.f;
      const int* idx = kSparse ? p.topk_idx + bt_row * p.topk : nullptr;
      for (int j = sg.t0; j < sg.t1; ++j, ++g) {
        const uint32_t sb = g & 1u, ph = (g >> 1) & 1u;
        const bool last = (j == sg.t1 - 1);
        ok = ok && warp_wait(bar(kSF + sb), ph, ctl);
        float s[32];
        if (ok) {
          tc_fence_after();
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + kColS + 64u * sb + 32u * half, r);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) s[c] = __uint_as_float(r[c]);
          tc_fence_before();
          mbar_arrive(bar(kSE + sb));
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) s[c] = NEG_INF;
        }

        // ---- mask (masked scores become -inf), then the row max of the raw
        // scores over both halves (the scale is positive, so max commutes with it)
        const int col0 = j * 64 + 32 * half;
        if (kSparse) {
          const bool vec = ((p.topk & 3) == 0) && ((reinterpret_cast<uintptr_t>(idx) & 15) == 0);
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            int iv[4];
            const int pos = col0 + 4 * c4;
            if (vec && pos + 3 < p.topk) {
              const int4 v = __ldg(reinterpret_cast<const int4*>(idx + pos));
              iv[0] = v.x; iv[1] = v.y; iv[2] = v.z; iv[3] = v.w;
            } else {
#pragma unroll
              for (int k = 0; k < 4; ++k) iv[k] = pos + k < p.topk ? __ldg(idx + pos + k) : -1;
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const bool valid = iv[k] >= 0 && iv[k] < L;
              s[4 * c4 + k] = valid ? s[4 * c4 + k] : NEG_INF;
            }
          }
        } else {
          const int nvalid = vis - col0;
          if (nvalid < 32) {
#pragma unroll
            for (int c = 0; c < 32; ++c) s[c] = c < nvalid ? s[c] : NEG_INF;
          }
        }
        float mh;
        {
          float m4[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
#pragma unroll
          for (int c = 0; c < 32; ++c) m4[c & 3] = fmaxf(m4[c & 3], s[c]);
          mh = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        }
        float* xm = xmax + (sb * 2) * kHeads;
        xm[half * kHeads + row] = mh;
        if (!named_bar_all(pair_bar, 64, ok)) {
          stop = true;
          break;
        }
        const float mt = fmaxf(mh, xm[(half ^ 1) * kHeads + row]) * p.scale_log2;  // same in both halves

        // ---- online softmax with a lazy rescale of the reference max
        float alpha = 1.f;
        if (mt > m_used + kRescaleLog2) {
          alpha = (m_used == NEG_INF) ? 0.f : ex2_approx(m_used - mt);
          m_used = mt;
          z *= alpha;
          zx *= alpha;
        }
        uint32_t pk[16];
        if (m_used == NEG_INF) {
#pragma unroll
          for (int c = 0; c < 16; ++c) pk[c] = 0u;
        } else {
          // P = 2^(s * scale_log2 - m) in one FFMA + EX2; the fp16-rounded
          // weights are widened exactly and summed in fp32
          float zs[4] = {0.f, 0.f, 0.f, 0.f}, ze[4] = {0.f, 0.f, 0.f, 0.f};
          const float nm = -m_used;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float p0 = ex2_approx(fmaf(s[2 * c], p.scale_log2, nm));
            const float p1 = ex2_approx(fmaf(s[2 * c + 1], p.scale_log2, nm));
            pk[c] = pack_f16x2(p0, p1);
            zs[c & 3] = add_f16x2_halves(zs[c & 3], pk[c]);
            ze[c & 3] += p0 + p1;
          }
          z += (zs[0] + zs[1]) + (zs[2] + zs[3]);
          zx += (ze[0] + ze[1]) + (ze[2] + ze[3]);
        }

        // ---- P message to the O side, once it is done with this slot
        ok = ok && warp_wait(bar(kPFree + sb), ph ^ 1u, ctl);
        const uint32_t mbar = rPM + 8u * sb;
        if (ok) {
          const uint32_t prow = rP + sb * kPBytes;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t piece = static_cast<uint32_t>(4 * half + k);
            st_async_v4(prow + ((piece ^ (row & 7)) << 4), pk[4 * k], pk[4 * k + 1], pk[4 * k + 2],
                        pk[4 * k + 3], mbar);
          }
          if (half == 0) st_async_b32(rAlpha + sb * kHeads * 4u, __float_as_uint(alpha), mbar);
        }
        if (last) {  // ---- segment end: both halves' sums -> final scale and LSE
          xsum[(half * 2 + 0) * kHeads + row] = z;
          xsum[(half * 2 + 1) * kHeads + row] = zx;
          if (!named_bar_all(pair_bar, 64, ok)) {
            stop = true;
            break;
          }
          if (half == 0) {
            const float zt = z + xsum[(2 + 0) * kHeads + row];
            const float zxt = zx + xsum[(2 + 1) * kHeads + row];
            const float fin = zt > 0.f ? 1.f / zt : 0.f;  // O_final = O_acc / z
            st_async_b32(rFin + sb * kHeads * 4u, __float_as_uint(fin), mbar);
            const float lse = zxt > 0.f ? (m_used + log2f(zxt)) * 0.69314718055994531f : NEG_INF;
            if (sg.slot < 0) {
              p.lse[bt_row * kHeads + row] = lse;
            } else if (sg.slot < 2 * U) {  // the plan never uses more than 2 * (U - 1) slots
              p.part_lse[(static_cast<long long>(sg.slot) * p.s_q + tok) * kHeads + row] = lse;
            }
          }
          if (!named_bar_all(pair_bar, 64, ok)) {  // xsum is reused at the next segment end
            stop = true;
            break;
          }
        }
      }
      ++nseg;
    }
  } else if (warp < 4) {
    // ================================================= O side: O correction + epilogue
    const int row = threadIdx.x;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const volatile float* alpha_s = reinterpret_cast<const volatile float*>(smem + kOffAlpha);
    const volatile float* fin_s = reinterpret_cast<const volatile float*>(smem + kOffFin);
    Seg64Iter<kPairTiles> it(p, unit);
    Seg sg;
    uint32_t g = 0, nseg = 0;
    bool ok = true;
    while (ok && it.next(sg)) {
      float fin = 0.f;
      for (int j = sg.t0; j < sg.t1; ++j, ++g) {
        const uint32_t pb = g & 1u, ph = (g >> 1) & 1u;
        const bool last = (j == sg.t1 - 1);
        if (row == 0) mbar_arrive_expect_tx(bar(kPM + pb), p_message_bytes(last));
        if (!(ok = __all_sync(0xffffffffu, wait_bar<true>(bar(kPM + pb), ph, ctl)))) break;
        const float alpha = alpha_s[pb * kHeads + row];
        if (last) fin = fin_s[pb * kHeads + row];
        const bool resc = (j != sg.t0) && alpha != 1.f;
        if (__any_sync(0xffffffffu, resc)) {  // tcgen05.ld/st are warp-collective
          // PV(g-1) finished: phase (g-1)/2 of the barrier of its parity (the
          // phase before it, PV(g-3), is known complete: P(g-1) was sent after it)
          const uint32_t gp = g - 1u;
          if (!(ok = warp_wait(bar(kPD + (gp & 1u)), (gp >> 1) & 1u, ctl))) break;
          tc_fence_after();
          const float a = resc ? alpha : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < 16; ++cc) {
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
        fence_proxy_async_smem();  // P written by st.async, read next by the tensor core
        tc_fence_before();
        mbar_arrive(bar(kPR + pb));

        if (last) {  // ---- segment epilogue: O * fin -> global
          if (!(ok = warp_wait(bar(kOF), nseg & 1u, ctl))) break;
          tc_fence_after();
          const long long bt_row = static_cast<long long>(sg.b) * p.s_q + tok;
          // final bf16 O, or a 16-bit partial (fp16: O of a split is a convex
          // combination of value rows, which the fp16 value product keeps
          // below 65504; bf16 with MLA_FLAG_BF16_PV), or final fp32 O
          const bool part = sg.slot >= 0;
          // rows are 1 or 2 KiB apart: 32-byte stores wherever the base allows
          // them (the workspace always does; the caller's output must be
          // 16-byte aligned only)
          const bool v8 = part || (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
          if (part && sg.slot >= 2 * U) {
            // the plan never uses more than 2 * (U - 1) slots
          } else if (part || !p.out_fp32) {
            uint16_t* dst0 = part
                ? p.part_o + ((static_cast<long long>(sg.slot) * p.s_q + tok) * kHeads + row) * kDv
                : static_cast<uint16_t*>(p.out) + (bt_row * kHeads + row) * kDv;
            const bool f16 = part && !p.part_bf16;
#pragma unroll 1
            for (int cc = 0; cc < 16; ++cc) {
              uint32_t r[32];
              tmem_ld32(tmem + lane_base + kColO + 32u * cc, r);
              tmem_wait_ld();
              uint4* dst = reinterpret_cast<uint4*>(dst0 + 32 * cc);
              uint32_t w[16];
              if (f16) {
#pragma unroll
                for (int c = 0; c < 16; ++c)
                  w[c] = pack_f16x2(__uint_as_float(r[2 * c]) * fin, __uint_as_float(r[2 * c + 1]) * fin);
              } else {
#pragma unroll
                for (int c = 0; c < 16; ++c)
                  w[c] = pack_bf16x2(__uint_as_float(r[2 * c]) * fin, __uint_as_float(r[2 * c + 1]) * fin);
              }
              if (v8) {  // whole 32-byte sectors
                st_global_v8(dst, w);
                st_global_v8(dst + 2, w + 8);
              } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) dst[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
              }
            }
          } else {
            float* dst0 = static_cast<float*>(p.out) + (bt_row * kHeads + row) * kDv;
#pragma unroll 1
            for (int cc = 0; cc < 16; ++cc) {
              uint32_t r[32];
              tmem_ld32(tmem + lane_base + kColO + 32u * cc, r);
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * fin);
              if (v8) {
#pragma unroll
                for (int k = 0; k < 4; ++k) st_global_v8(dst0 + 32 * cc + 8 * k, r + 8 * k);
              } else {
                float4* dst = reinterpret_cast<float4*>(dst0 + 32 * cc);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                  dst[k] = make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                                       __uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3]));
              }
            }
          }
          tc_fence_before();
          mbar_arrive(bar(kOE));
        }
      }
      ++nseg;
    }
  } else if (warp == 8) {
    // ================================================= MMA issue (one thread)
    if (lane == 0) {
      Seg64Iter<kPairTiles> it(p, unit);
      Seg sg;
      Ring3 rs;
      uint32_t g = 0, nseg = 0;
      bool ok = true;
      while (ok && it.next(sg)) {
        if (s_side) {
          // Q of this segment arrives as three ring slots of three 64-dim chunks
          // (16 KiB each, 128-byte swizzled); tcgen05.cp moves them into TMEM
          // once the previous segment's score MMAs have read the old Q
          if (nseg > 0 && !(ok = wait_bar<false>(bar(kQF), (nseg - 1u) & 1u, ctl))) break;
          for (int k = 0; k < 3 && ok; ++k, rs.advance()) {
            if (!(ok = wait_bar<false>(bar((kFp8 ? kVR : kKF) + rs.idx), rs.phase, ctl))) break;
            tc_fence_after();
            const uint64_t qd0 = smem_desc(sStage + rs.idx * stage_bytes, 16u, 1024u);
#pragma unroll
            for (int i = 0; i < 3; ++i) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                tmem_cp_128x256b(tmem + kColQ + 32u * (3 * k + i) + 8u * kk,
                                 qd0 + static_cast<uint64_t>((i * kQChunkBytes + 32 * kk) >> 4));
            }
            umma_commit(bar(kKE + rs.idx));
          }
          if (!ok) break;
        }
        for (int j = sg.t0; j < sg.t1; ++j, ++g, rs.advance()) {
          const uint32_t stg = sStage + rs.idx * stage_bytes;
          const uint32_t sb = g & 1u, ph = (g >> 1) & 1u;
          if (s_side) {
            // the tile landed (bf16), or was widened by the fill threads (FP8)
            if (!(ok = wait_bar<false>(bar((kFp8 ? kVR : kKF) + rs.idx), rs.phase, ctl))) break;
            if (kSparse) fence_proxy_async_smem();  // rows written by the gather threads' copies
            if (!(ok = wait_bar<false>(bar(kSE + sb), ph ^ 1u, ctl))) break;
            tc_fence_after();
            // 36 MMAs (K = 576 in steps of 16): descriptors differ from the
            // tile's base descriptor by compile-time offsets
            const uint64_t bd0 = smem_desc(stg, 16u, 1024u);
            const uint32_t dS = tmem + kColS + 64u * sb;
#pragma unroll
            for (int c = 0; c < kNumChunks; ++c) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_f16_tmem_a(dS, tmem + kColQ + 32u * c + 8u * kk,
                                bd0 + static_cast<uint64_t>((c * kChunkBytes + 32 * kk) >> 4),
                                (kFp8 && c < 8) ? kIdescQK16 : kIdescQK,
                                (c | kk) != 0 ? 1u : 0u);
            }
            umma_commit(bar(kSF + sb));
            umma_commit(bar(kKE + rs.idx));
            if (j == sg.t1 - 1) umma_commit(bar(kQF));
          } else {
            const bool first = (j == sg.t0);
            if (!(ok = wait_bar<false>(bar(kVR + rs.idx), rs.phase, ctl))) break;
            if (!(ok = wait_bar<false>(bar(kPR + sb), ph, ctl))) break;
            if (first && !(ok = wait_bar<false>(bar(kOE), (nseg & 1u) ^ 1u, ctl))) break;
            tc_fence_after();
            const uint64_t ad0 = smem_desc(sP + sb * kPBytes, 16u, 1024u);
            const uint64_t bd0 = smem_desc(stg, 8192u, 1024u);  // V, MN-major
            const uint32_t acc0 = first ? 0u : 1u;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
              for (int h = 0; h < 2; ++h)
                umma_f16(tmem + kColO + 256u * h, ad0 + static_cast<uint64_t>((32 * kk) >> 4),
                         bd0 + static_cast<uint64_t>((h * 4 * kChunkBytes + 2048 * kk) >> 4), kIdescPV,
                         kk == 0 ? acc0 : 1u);
            }
            umma_commit(bar(kKE + rs.idx));
            umma_commit_multicast(bar(kPFree + sb), 1);  // the S side may reuse this P slot
            umma_commit(bar(kPD + sb));
            if (j == sg.t1 - 1) umma_commit(bar(kOF));
          }
        }
        ++nseg;
      }
      umma_commit(bar(kMmaDone));  // every MMA issued so far has finished before TMEM goes
      drain_bar(bar(kMmaDone), 0);
    }
    __syncwarp();
  } else if (warp == 9 && !kSparse) {
    // ================================================= TMA producer (whole warp; lane 0 issues)
    // S side: per segment three Q slots, then (dense) one slot per tile.  O
    // side (dense): one slot per tile, value dims only.  Page ids are read 32
    // at a time with one coalesced load.  (No L2 prefetch from this SM: it
    // would share the TMA unit with the loads and delay them.)
    Seg64Iter<kPairTiles> it(p, unit);
    Seg sg;
    Ring3 rs;
    uint32_t issued = 0;
    bool ok = true;
    // in sparse mode the gather warps are the only filler of the ring (the S
    // side's gather warps load Q too): a ring shared by two fillers could let
    // one of them drift a whole lap, which mbarrier parity waits cannot see
    while (!kSparse && ok && it.next(sg)) {
      if (s_side) {
        const int qy = (sg.b * p.s_q + tok) * kHeads;
        for (int k = 0; k < 3 && ok; ++k, rs.advance()) {
          if (!(ok = warp_wait(bar(kKE + rs.idx), rs.phase ^ 1u, ctl))) break;
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(kKF + rs.idx), 3 * kQChunkBytes);
            for (int i = 0; i < 3; ++i)
              tma_load_2d(sStage + rs.idx * stage_bytes + i * kQChunkBytes, &tm_q, (3 * k + i) * kChunk, qy,
                          bar(kKF + rs.idx));
          }
          ++issued;
        }
        if (!ok) break;
      }
      const int* bt_row = p.block_table + static_cast<long long>(sg.b) * p.bt_stride;
      for (int jb = sg.t0; jb < sg.t1 && ok; jb += 32) {
        const int cnt = min(32, sg.t1 - jb);
        int my_page = -1;
        if (lane < cnt && jb + lane < p.bt_stride) {
          const int pg = bt_row[jb + lane];
          my_page = (pg >= 0 && pg < p.num_pages) ? pg : -1;
        }
        for (int jj = 0; jj < cnt; ++jj, rs.advance()) {
          const int page = __shfl_sync(0xffffffffu, my_page, jj);
          if (!(ok = warp_wait(bar(kKE + rs.idx), rs.phase ^ 1u, ctl))) break;
          if (lane == 0) {
            // an entry outside the pool reads the TMA fill value (zeros)
            const int y = page >= 0 ? page * kPage : static_cast<int>(p.num_pages) * kPage;
            const uint32_t stg = sStage + rs.idx * stage_bytes;
            if (kFp8) {  // latent + scale bytes to the stage's end; the S side's RoPE chunk to chunk 8
              mbar_arrive_expect_tx(bar(kKF + rs.idx), kF8RawBytes + (s_side ? kChunkBytes : 0));
              tma_load_2d(stg + kF8RawOff, &tm_kv, 0, y, bar(kKF + rs.idx));
              if (s_side) tma_load_2d(stg + 8 * kChunkBytes, &tm_rope, kF8Lat / 2, y, bar(kKF + rs.idx));
            } else {  // the tile's nine (S side) or eight (O side) chunks as one 3-D box
              mbar_arrive_expect_tx(bar(kKF + rs.idx), nchunks * kChunkBytes);
              tma_load_3d(stg, s_side ? &tm_kv : &tm_rope, 0, y, 0, bar(kKF + rs.idx));
            }
          }
          ++issued;
        }
      }
    }
    if (!ok && lane == 0) {  // let copies in flight land before the CTA goes away
      for (uint32_t k = 0; k < static_cast<uint32_t>(kStages) && k < issued; ++k) {
        const uint32_t t = issued - 1 - k;
        drain_bar(bar(kKF + t % kStages), (t / kStages) & 1u);
      }
    }
  } else {
    // ================================================= O side warps 4-7 (+10-11 dense): V conversion
    // (dense) or gather + conversion (sparse); S side warps 10-11: gather (sparse)
    // dense: O side warps 4-7, 10-11 convert (ptid 0..191); sparse: S side
    // warps 9-19 (ptid 0..351) and O side warps 4-7, 10-19 (0..447) gather
    const int ptid = s_side ? threadIdx.x - 288 : (warp < 8 ? threadIdx.x - 128 : threadIdx.x - 192);
    Seg64Iter<kPairTiles> it(p, unit);
    Seg sg;
    Ring3 rs;
    bool ok = true;
    if (kFp8) {
      if (!(kSparse && !s_side && warp == 9)) {
        // ---- FP8 cache: fill threads widen each tile's codes in place
        const int nthreads = f8_fill_threads(kSparse, s_side);
        const int fid = s_side ? threadIdx.x - (kSparse ? 288 : 320) : ptid;  // 0 .. nthreads - 1
        const uint8_t* kv8 = reinterpret_cast<const uint8_t*>(p.kv);
        // Stage `stg`'s raw bytes (64 rows x 528 at kF8RawOff) -> fp16
        // chunks 0-7 (the S side's RoPE chunk 8 stays bf16).  Raw piece
        // P (16 codes) is row (P >> 2) & 63, dims 64 (P >> 8) + 16 (P & 3) ..;
        // its output is pieces 2 (P & 3) and 2 (P & 3) + 1 of that row in
        // chunk P >> 8.  Rows >= r_end are written as zeros.  Chunks 0-2 end
        // below the raw bytes and are written as they are read; chunks 3-7
        // overwrite them, so every thread reads its pieces of those first and
        // writes them after the group barrier (which also votes `ok`, the
        // result returned).
        auto convert = [&](uint32_t stg, int r_end, bool ok_in) -> bool {
          const uint32_t raw = stg + kF8RawOff;
          // widen raw piece P (codes v, scale byte E) and store its two output pieces
          auto put = [&](int P, uint4 v, uint32_t E) {
            const int r = (P >> 2) & 63;
            const uint32_t h = static_cast<uint32_t>(P & 3);
            const uint32_t o = stg + static_cast<uint32_t>((P >> 8) * kChunkBytes + r * 128);
            const uint32_t sw = static_cast<uint32_t>(r & 7);
            if (r >= r_end) {
              st_shared_zero16(o + (((2u * h) ^ sw) << 4));
              st_shared_zero16(o + (((2u * h + 1u) ^ sw) << 4));
            } else {
              uint32_t w[8];
              widen_f16(v, f16_scale_pair(E), w);
              st_shared_v4(o + (((2u * h) ^ sw) << 4), w[0], w[1], w[2], w[3]);
              st_shared_v4(o + (((2u * h + 1u) ^ sw) << 4), w[4], w[5], w[6], w[7]);
            }
          };
          auto raw_piece = [&](int P, uint4& v, uint32_t& E) {
            const uint32_t rb = raw + static_cast<uint32_t>(((P >> 2) & 63) * kF8Lat);
            v = ld_shared_v4u(rb + static_cast<uint32_t>(64 * (P >> 8) + 16 * (P & 3)));
            E = ld_shared_u8(rb + 512u + static_cast<uint32_t>(P >> 9));
          };
          // chunks 3-7 overwrite raw bytes: this thread's pieces of them are
          // read first, and written only after the group barrier
          uint4 v[kF8PerThread];
          uint32_t e[kF8PerThread];
#pragma unroll
          for (int k = 0; k < kF8PerThread; ++k) {
            const int P = kF8Low + fid + nthreads * k;
            if (P < kF8Pieces) raw_piece(P, v[k], e[k]);
          }
          // chunks 0-2 lie below the raw bytes: streamed before the barrier
#pragma unroll 2
          for (int P = fid; P < kF8Low; P += nthreads) {
            uint4 c;
            uint32_t E;
            raw_piece(P, c, E);
            put(P, c, E);
          }
          if (!named_bar_all(5, nthreads, ok_in)) return false;
#pragma unroll
          for (int k = 0; k < kF8PerThread; ++k) {
            const int P = kF8Low + fid + nthreads * k;
            if (P < kF8Pieces) put(P, v[k], e[k]);
          }
          fence_proxy_async_smem();  // generic writes, read next by the tensor core
          return true;
        };
        if (!kSparse) {
          // dense: warp 9 loads (TMA); the fill threads pass Q slots on and
          // widen each tile (the O side zeroes rows past the cache end)
          while (ok && it.next(sg)) {
            if (s_side) {
              for (int k = 0; k < 3; ++k, rs.advance()) {
                ok = ok && warp_wait(bar(kKF + rs.idx), rs.phase, ctl);
                if (ok) {  // Q's latent dims (bf16) -> fp16; its RoPE chunk (8, in slot 2) stays bf16
                  bf16_region_to_f16(sStage + rs.idx * stage_bytes, fid, nthreads, (k < 2 ? 3 : 2) * kQChunkBytes / 16);
                  fence_proxy_async_smem();
                  mbar_arrive(bar(kVR + rs.idx));
                }
              }
            }
            const int L = max(p.cache_lens[sg.b], 0);
            for (int j = sg.t0; j < sg.t1; ++j, rs.advance()) {
              ok = ok && warp_wait(bar(kKF + rs.idx), rs.phase, ctl);
              if (!(ok = convert(sStage + rs.idx * stage_bytes, s_side ? kPage : L - j * 64, ok))) break;
              mbar_arrive(bar(kVR + rs.idx));
            }
          }
        } else {
          // top-k: the fill threads gather the named rows' latent + scale
          // bytes (and on the S side the RoPE dims, straight into chunk 8)
          // with 16-byte cp.async copies, one row per warp at a time, and
          // widen tile j - 1 after issuing tile j's copies.  Rows the list
          // does not name (or outside the pool) are zero-filled: value 0.
          const int nw = nthreads / 32;
          const int gw = fid >> 5;
          const int rows_w = (kPage - gw + nw - 1) / nw;
          const int npc = s_side ? kF8Lat / 16 + 8 : kF8Lat / 16;  // 16-byte pieces per row
          int pend = -1;
          // kKF completes only for the Q slots here (tiles land by cp.async):
          // the parity of its next phase is tracked per slot, not by the ring
          uint32_t qpar = 0u;
          while (ok && it.next(sg)) {
            if (s_side) {  // three Q slots (TMA from one fill thread), passed on once landed
              for (int k = 0; k < 3; ++k, rs.advance()) {
                ok = ok && warp_wait(bar(kKE + rs.idx), rs.phase ^ 1u, ctl);
                if (ok && fid == 0) {
                  const int qy = (sg.b * p.s_q + tok) * kHeads;
                  mbar_arrive_expect_tx(bar(kKF + rs.idx), 3 * kQChunkBytes);
                  for (int i = 0; i < 3; ++i)
                    tma_load_2d(sStage + rs.idx * stage_bytes + i * kQChunkBytes, &tm_q, (3 * k + i) * kChunk, qy,
                                bar(kKF + rs.idx));
                }
                ok = ok && warp_wait(bar(kKF + rs.idx), (qpar >> rs.idx) & 1u, ctl);
                qpar ^= 1u << rs.idx;
                if (ok) {  // Q's latent dims (bf16) -> fp16; its RoPE chunk (8, in slot 2) stays bf16
                  bf16_region_to_f16(sStage + rs.idx * stage_bytes, fid, nthreads, (k < 2 ? 3 : 2) * kQChunkBytes / 16);
                  fence_proxy_async_smem();
                  mbar_arrive(bar(kVR + rs.idx));
                }
              }
            }
            const int L = max(p.cache_lens[sg.b], 0);
            const long long bt_row = static_cast<long long>(sg.b) * p.s_q + tok;
            const int* idx = p.topk_idx + bt_row * p.topk;
            const int* tbl = p.block_table + static_cast<long long>(sg.b) * p.bt_stride;
            auto lookup = [&](int j) -> long long {
              long long pr = -1;
              if (lane < rows_w) {
                const int pos = j * 64 + gw + nw * lane;
                if (pos < p.topk) {
                  const int ix = __ldg(idx + pos);
                  if (ix >= 0 && ix < L && (ix >> 6) < p.bt_stride) {
                    const int pg = __ldg(tbl + (ix >> 6));
                    if (pg >= 0 && pg < p.num_pages) pr = static_cast<long long>(pg) * kPage + (ix & 63);
                  }
                }
              }
              return pr;
            };
            long long my_row = lookup(sg.t0);
            for (int j = sg.t0; j < sg.t1; ++j, rs.advance()) {
              ok = ok && warp_wait(bar(kKE + rs.idx), rs.phase ^ 1u, ctl);
              if (!(ok = named_bar_all(5, nthreads, ok))) break;
              const uint32_t stg = sStage + rs.idx * stage_bytes;
              for (int i = 0; i < rows_w; ++i) {
                const long long prow = __shfl_sync(0xffffffffu, my_row, i);
                const int r = gw + nw * i;
                const uint8_t* src = kv8 + (prow >= 0 ? prow : 0) * kF8Row;
                const uint32_t src_bytes = prow >= 0 ? 16u : 0u;  // 0: the copy writes zeros
                for (int c16 = lane; c16 < npc; c16 += 32) {
                  if (c16 < kF8Lat / 16) {
                    cp_async_16_zfill(stg + kF8RawOff + r * kF8Lat + 16 * c16, src + 16 * c16, src_bytes);
                  } else {
                    const int q = c16 - kF8Lat / 16;  // RoPE piece q -> chunk 8, swizzled
                    cp_async_16_zfill(stg + 8 * kChunkBytes + r * 128 + ((q ^ (r & 7)) << 4), src + kF8Lat + 16 * q,
                                      src_bytes);
                  }
                }
              }
              if (j + 1 < sg.t1) my_row = lookup(j + 1);
              cp_async_commit();
              if (pend >= 0) {  // the previous tile: every thread's copies landed -> widen
                cp_async_wait<1>();
                named_bar_sync(5, nthreads);
                if (!(ok = convert(sStage + pend * stage_bytes, kPage, ok))) break;
                mbar_arrive(bar(kVR + pend));
              }
              pend = static_cast<int>(rs.idx);
            }
            if (ok && pend >= 0) {  // the segment's last tile
              cp_async_wait<0>();
              named_bar_sync(5, nthreads);
              if (!(ok = convert(sStage + pend * stage_bytes, kPage, ok))) break;
              mbar_arrive(bar(kVR + pend));
              pend = -1;
            }
          }
          cp_async_wait<0>();  // no copy outlives the CTA
        }
      }
    } else if ((!kSparse && s_side) || (kSparse && !s_side && warp == 9)) {
      // nothing to do: the S side consumes TMA tiles as they land
    } else if (!kSparse) {
      // ---- O side, dense: 192 threads convert the landed bf16 value tile to fp16 in place
      constexpr int kPieces = kStageO / 16;  // 4096 pieces of 16 B
      while (ok && it.next(sg)) {
        const int L = max(p.cache_lens[sg.b], 0);
        for (int j = sg.t0; j < sg.t1; ++j, rs.advance()) {
          if (!(ok = warp_wait(bar(kKF + rs.idx), rs.phase, ctl))) break;
          const uint32_t stg = sStage + rs.idx * kStageO;
          const int r_end = L - j * 64;  // rows >= r_end lie past the cache end: zero them
          if (r_end >= 64) {
#pragma unroll 4
            for (int piece = ptid; piece < kPieces; piece += conv_threads(false)) {
              const uint32_t a = stg + 16u * piece;
              uint4 v;
              asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
              st_shared_v4(a, bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z),
                           bf16x2_to_f16x2(v.w));
            }
          } else {
            for (int piece = ptid; piece < kPieces; piece += conv_threads(false)) {
              const uint32_t a = stg + 16u * piece;
              const int r = (piece & 511) >> 3;  // the swizzle only permutes pieces within a row
              if (r >= r_end) {
                st_shared_zero16(a);
              } else {
                uint4 v;
                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
                st_shared_v4(a, bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z),
                             bf16x2_to_f16x2(v.w));
              }
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(bar(kVR + rs.idx));
        }
      }
    } else {
      // ---- sparse: rows named by the index list are gathered with 16-byte
      // cp.async copies, one row at a time per warp so that a warp's copies
      // read contiguous bytes (a lane per 16-byte piece): on the S side eleven
      // warps (all 576 dims), on the O side fourteen (the 512 value dims, which
      // they then convert to fp16 in place); warp w of n takes rows w, w + n,
      // ...  Rows the list does not name (or that lie outside the pool) are
      // zero-filled.  Each lane looks up one row's pool position, a tile
      // ahead, and the warp shares them by shuffles.  Nothing waits for a
      // tile's copies where they are issued: on the S side the tile's landing
      // barrier tracks every gather thread's copies (the MMA thread then
      // orders them before its tensor-core reads); on the O side a warp
      // converts tile j - 1 after issuing tile j's copies.
      const int nthreads = s_side ? 352 : conv_threads(true);
      const int nw = nthreads / 32;
      const int gw = ptid >> 5;                          // gather warp 0 .. nw - 1
      const int rows_w = (kPage - gw + nw - 1) / nw;     // rows gw, gw + nw, ... of a tile
      const int npc = s_side ? kNumChunks * 8 : 64;      // 16-byte pieces per row
      // O side: convert the pieces this lane brought into stage `st`
      auto convert_own = [&](uint32_t st) {
        for (int i = 0; i < rows_w; ++i) {
          const int r = gw + nw * i;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int c16 = lane + 32 * k;
            const uint32_t a = st + (c16 >> 3) * kChunkBytes + r * 128 + (((c16 & 7) ^ (r & 7)) << 4);
            const uint4 v = ld_shared_v4u(a);
            st_shared_v4(a, bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z),
                         bf16x2_to_f16x2(v.w));
          }
        }
      };
      int pend = -1;  // O side: stage index of the tile whose copies are still in flight
      while (ok && it.next(sg)) {
        if (s_side) {  // three Q slots (TMA, issued by one gather thread)
          const int qy = (sg.b * p.s_q + tok) * kHeads;
          for (int k = 0; k < 3 && ok; ++k, rs.advance()) {
            if (!(ok = warp_wait(bar(kKE + rs.idx), rs.phase ^ 1u, ctl))) break;
            if (ptid == 0) {
              mbar_arrive_expect_tx(bar(kKF + rs.idx), 3 * kQChunkBytes);
              for (int i = 0; i < 3; ++i)
                tma_load_2d(sStage + rs.idx * stage_bytes + i * kQChunkBytes, &tm_q, (3 * k + i) * kChunk, qy,
                            bar(kKF + rs.idx));
            }
          }
          if (!ok) break;
        }
        const int L = max(p.cache_lens[sg.b], 0);
        const long long bt_row = static_cast<long long>(sg.b) * p.s_q + tok;
        const int* idx = p.topk_idx + bt_row * p.topk;
        const int* tbl = p.block_table + static_cast<long long>(sg.b) * p.bt_stride;
        // this lane's row of the warp's share of tile j: its pool row, or -1
        auto lookup = [&](int j) -> long long {
          long long pr = -1;
          if (lane < rows_w) {
            const int pos = j * 64 + gw + nw * lane;
            if (pos < p.topk) {
              const int ix = __ldg(idx + pos);
              if (ix >= 0 && ix < L && (ix >> 6) < p.bt_stride) {
                const int pg = __ldg(tbl + (ix >> 6));
                if (pg >= 0 && pg < p.num_pages) pr = static_cast<long long>(pg) * kPage + (ix & 63);
              }
            }
          }
          return pr;
        };
        long long my_row = lookup(sg.t0);
        for (int j = sg.t0; j < sg.t1; ++j, rs.advance()) {
          ok = warp_wait(bar(kKE + rs.idx), rs.phase ^ 1u, ctl);
          // the S side's gather warps meet at a named barrier below: they vote
          // here so that all leave if any wait ran out
          if (s_side) ok = named_bar_all(5, nthreads, ok);
          if (!ok) break;
          const uint32_t stg = sStage + rs.idx * stage_bytes;
          for (int i = 0; i < rows_w; ++i) {
            const long long prow = __shfl_sync(0xffffffffu, my_row, i);
            const int r = gw + nw * i;
            const uint16_t* src = p.kv + (prow >= 0 ? prow : 0) * kDqk;
            const uint32_t src_bytes = prow >= 0 ? 16u : 0u;  // 0: the copy writes zeros
            for (int c16 = lane; c16 < npc; c16 += 32)
              cp_async_16_zfill(stg + (c16 >> 3) * kChunkBytes + r * 128 + (((c16 & 7) ^ (r & 7)) << 4),
                                src + c16 * 8, src_bytes);
          }
          if (j + 1 < sg.t1) my_row = lookup(j + 1);  // its latency overlaps the copies and the next wait
          if (s_side) {
            cp_async_mbar_track(bar(kKF + rs.idx));
            named_bar_sync(5, nthreads);  // every thread's copies are tracked before the one arrival
            if (ptid == 0) mbar_arrive(bar(kKF + rs.idx));
          } else {
            cp_async_commit();
            if (pend >= 0) {  // the previous tile: landed -> fp16 -> ready for the value product
              cp_async_wait<1>();
              convert_own(sStage + pend * stage_bytes);
              fence_proxy_async_smem();
              mbar_arrive(bar(kVR + pend));
            }
            pend = static_cast<int>(rs.idx);
          }
        }
        if (!s_side && pend >= 0 && ok) {  // the segment's last tile
          cp_async_wait<0>();
          convert_own(sStage + pend * stage_bytes);
          fence_proxy_async_smem();
          mbar_arrive(bar(kVR + pend));
          pend = -1;
        }
      }
      cp_async_wait<0>();  // no copy outlives the CTA
    }
  }

  // ======================================================= teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer no longer touches this CTA's shared memory
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
int decode_smem_bytes() { return kSmemBytes; }
int decode_threads(bool sparse, bool fp8) { return fp8 ? kThreadsFp8 : (sparse ? kThreadsSparse : kThreads); }

cudaError_t decode_set_attrs() {
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel<false, false>, a, kSmemBytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(mla_decode_kernel<true, false>, a, kSmemBytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(mla_decode_kernel<false, true>, a, kSmemBytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(mla_decode_kernel<true, true>, a, kSmemBytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(mla_decode_kernel<false, true, true>, a, kSmemBytes);
  return e;
}

// `dependent`: may be scheduled while the previous kernel on the stream (the
// plan) finishes (programmatic dependent launch).
static void cluster_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int num_clusters,
                           cudaStream_t stream, int threads, bool dependent) {
  cfg = cudaLaunchConfig_t{};
  cfg.gridDim = dim3(2 * num_clusters, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;  // the kernel always runs as CTA pairs
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 2 : 1;
}

// Co-resident 2-CTA clusters of the decode kernel on the current device.
cudaError_t decode_max_clusters(int* n, int num_clusters_hint) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  cluster_config(cfg, attr, num_clusters_hint, nullptr, decode_threads(false, false), false);
  return cudaOccupancyMaxActiveClusters(n, mla_decode_kernel<false, false>, &cfg);
}

// Maps: bf16 cache, tm_kv = a page's nine chunks (S side), tm_rope = its
// eight value chunks (O side), as 3-D boxes; FP8 cache, tm_kv = each row's
// 528 latent + scale bytes, tm_rope = its 64 bf16 RoPE dims.
cudaError_t decode_launch(bool sparse, bool fp8, bool pair_tiles, int num_clusters, cudaStream_t stream,
                          const DecodeParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_kv,
                          const CUtensorMap& tm_rope) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  cluster_config(cfg, attr, num_clusters, stream, decode_threads(sparse, fp8), true);
  if (fp8 && pair_tiles)  // two query tokens over a dense FP8 cache (plan tiles of 128 rows)
    return cudaLaunchKernelEx(&cfg, mla_decode_kernel<false, true, true>, p, tm_q, tm_kv, tm_rope);
  if (fp8)
    return sparse ? cudaLaunchKernelEx(&cfg, mla_decode_kernel<true, true>, p, tm_q, tm_kv, tm_rope)
                  : cudaLaunchKernelEx(&cfg, mla_decode_kernel<false, true>, p, tm_q, tm_kv, tm_rope);
  return sparse ? cudaLaunchKernelEx(&cfg, mla_decode_kernel<true, false>, p, tm_q, tm_kv, tm_rope)
                : cudaLaunchKernelEx(&cfg, mla_decode_kernel<false, false>, p, tm_q, tm_kv, tm_rope);
}

}  // namespace mla
