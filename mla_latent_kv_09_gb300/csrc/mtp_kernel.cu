// mtp_kernel.cu — MLA decode for requests with two query tokens (s_q = 2,
// the multi-token-prediction step) on sm_103a, with paired-SM tensor-core
// operations.
//
// What it computes is the attention of decode_kernel.cu ("DeepSeek V3/R1
// Inference Efficiency (2)", §2.4.1, "MLA/MQA attention"); under the causal
// mask the second token sees one more cached position than the first.  Both
// tokens of a request read the same pages, so one tile of cached rows serves
// both, and their 2 x 128 query heads form one M = 256 operand of a tcgen05
// operation spread over a pair of SMs (cta_group::2: each SM of the pair holds
// half of the rows of A and D and half of the columns of B).
//
// One work unit = one 4-CTA cluster = two SM pairs.  A tile is 128 cached
// rows (two pages).
//   Ranks 0, 1 (score pair).  Rank r holds token r's Q — dims 0..511 in tensor
//     memory, the 64 RoPE dims in shared memory — and streams page r of every
//     tile (all 576 dims) through a ring of 21 chunk slots of 8 KiB, freed
//     and refilled in groups of three as soon as the score MMAs reading them
//     finish; Q dims 0..511 come through the same ring (and tcgen05.cp) at the
//     start of each segment.  Rank 0 issues S = Q K^T for both tokens (M =
//     256, N = 128, K = 576) into two alternating 128-column score buffers;
//     token r's rows land in rank r.  Each rank runs the online softmax of
//     its token (fp32, exp2 domain, lazy rescale: the reference max moves
//     only when a score beats it by more than 2^8) and sends P plus the
//     per-row rescale factor to rank 2 + r.
//   Ranks 2, 3 (value pair).  Rank 2 + r owns token r's O (128 x 512 fp32,
//     all of its tensor memory).  Rank 2 + r loads the value dims
//     [128 r, 128 r + 128) and [256 + 128 r, 256 + 128 r + 128) of both pages
//     (the B columns it holds in the pair) through a ring of page slots, and
//     rank 2 issues O += P V (M = 256, N = 2 x 256, K = 128).  At the end of
//     a segment all sixteen warps write O (scaled by 1 / z) with tensor
//     stores, staged in the P slot the last tile used.
// P and V are fp16 by default (11 significant bits on the softmax weights;
// values must stay below 65504 in magnitude): the value ranks' conversion
// warps read each page's value dims from global memory (an L2 hit behind the
// score ranks' loads), convert them and store them into the page slot, each
// warp announcing its rows to rank 2 itself.  The kBf16PV variant (bf16 P and
// V, on request) loads the value dims with TMA instead.
//
// Warps (640 threads).  Score ranks: 0-15 softmax (warp w: head rows
// 32 (w % 4) .., key columns 32 (w / 4) .. of each tile), 16 and 19 MMA issue
// on rank 0 (even and odd tiles; 16 also owns tensor memory and moves Q in),
// 17 TMA producer, 18 P shipper.  Value ranks: 0-3 O rescale (thread i = head
// row i), 4-15 V conversion (fp16 variant; rows past the cache end are zeroed
// in both), 0-15 the segment epilogue, 16 MMA issue on rank 2 and
// tensor-memory owner, 17 TMA producer.
//
// Two threads issue the score MMAs, alternating tiles: one thread issues
// these paired MMAs at ~73-110 cycles each while the pipe executes one every
// 64, so the pipe is full only while both issue.  Each issuer waits for its
// tile's score buffer (freed by every softmax warp right after its own
// tensor-memory load) and first slot group while the other issues, takes an
// issue token from the other, issues its 36 MMAs — probing the next slot
// group without blocking a few MMAs ahead — and passes the token on after
// 24 MMAs.
//
// P travels as one bulk copy per tile: the softmax warps write it into a
// local copy laid out as the value rank's A operand; the shipper warp sends
// it with cp.async.bulk (completing on the value rank's barrier) once PV is
// done with the destination slot, and frees the local copy when the bulk copy
// has read it.  Shared-memory-to-shared-memory traffic between SMs is the
// narrowest path of this kernel (about 21 B per clock per SM), so the softmax
// warps never wait for it except when they are a whole tile ahead.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernel_common.cuh"
#include "plan.cuh"
#include "ptx.cuh"

namespace mla {
namespace mtp {

// Arrive on an mbarrier of the value pair's rank 2 with release at CTA scope:
// the arriving warp's shared-memory stores are performed before the arrive
// lands.  The tensor core of the pair reads them from this CTA's shared memory
// only after rank 2 has seen the arrival.  (Release at cluster scope costs
// each arriving warp about a thousand cycles under load.)
__device__ __forceinline__ void mbar_arrive_remote_cta(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}

constexpr int kTileRows = 2 * kPage;              // 128 cached rows per tile
constexpr int kPageChunk = kPage * 128;           // 8 KiB: 64 rows x 64 dims (bf16), 128B-swizzled
constexpr int kKSlots = 21;                       // score ranks: chunk slots (2 1/3 tiles)
constexpr int kKGroup = 3;                        // chunk slots per landing / free barrier
constexpr int kKGroups = kKSlots / kKGroup;
constexpr int kVPage = 4 * kPageChunk;            // 32 KiB: one page, this rank's 256 value dims
constexpr int kVSlots = 4;                        // value ranks: page slots (two tiles)
constexpr int kVDepth = 1;                        // fp16 variant: pages of value loads in flight per thread
                                                  // beyond the one being stored (2 measured no faster)
// P tile, 128 heads x 128 keys of 16-bit weights, as a K-major 128B-swizzled
// operand whose 8-row groups hold both 64-key halves side by side: byte
// (row / 8) * 2048 + half * 1024 + (row % 8) * 128 + swizzled 16-B piece.  A
// row quarter (32 rows) is then one contiguous 8 KiB block.
constexpr int kPSlot = kHeads * 256;              // 32 KiB
constexpr int kPGroupStride = 2048;               // between 8-row groups
constexpr int kPHalfStride = 1024;                // between the two 64-key halves
constexpr int kQChunk = kHeads * 128;             // 16 KiB: 128 heads x 64 dims (bf16)

// Shared memory (offsets from a 1024-aligned base; the barrier block sits at
// the same offset in all four CTAs, which multicast commits rely on).
constexpr int kOffStage = 0;                         // chunk slots (score ranks) / page slots (value ranks)
constexpr int kOffQr = kKSlots * kPageChunk;         // score ranks: Q dims 512..575
constexpr int kOffXchg = kOffQr + kQChunk;           // score ranks: row max / sums exchange, 8 KiB
constexpr int kOffPs = kOffXchg + 8192;              // score ranks: outgoing P tile (same layout as kOffP)
constexpr int kOffAlphaS = kOffPs + kPSlot;          // score ranks: outgoing float[128] rescale factors
constexpr int kOffFinS = kOffAlphaS + kHeads * 4;    // score ranks: outgoing float[128] final scales
constexpr int kEndS = kOffFinS + kHeads * 4;         // 230400
constexpr int kOffP = kVSlots * kVPage;              // value ranks: [2] P tiles
constexpr int kOffAlpha = kOffP + 2 * kPSlot;        // value ranks: float[2][128]
constexpr int kOffFin = kOffAlpha + 2 * kHeads * 4;  // value ranks: float[2][128]
constexpr int kEndO = kOffFin + 2 * kHeads * 4;      // 198656
constexpr int kOffBar = kEndS > kEndO ? kEndS : kEndO;
constexpr int kBarBytes = 640;
constexpr int kAlignSlack = 1024;
constexpr int kSmemBytes = kOffBar + kBarBytes + kAlignSlack;
static_assert(kOffPs % 1024 == 0 && kOffP % 1024 == 0, "P tiles keep the 128-byte swizzle phase");
static_assert(kSmemBytes <= 232448, "shared memory");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // score ranks: two 128-column score buffers
constexpr uint32_t kColQ = 256;  // score ranks: Q dims 0..511, 8 chunks of 32 columns
constexpr uint32_t kColO = 0;    // value ranks: O, 512 columns

constexpr int kThreads = 640;                    // 20 warps
constexpr int kSoftmaxWarps = 16;
constexpr int kConvThreads = 384;                // value ranks: warps 4-15
constexpr int kMmaWarp = 16;
constexpr int kTmaWarp = 17;
constexpr int kShipWarp = 18;                    // score ranks: P shipper
constexpr int kMma2Warp = 19;                    // rank 0: issues the score MMAs of odd tiles
constexpr float kRescaleLog2 = 8.0f;

constexpr uint16_t kScoreMask = 0x3;  // ranks 0, 1
constexpr uint16_t kValueMask = 0xC;  // ranks 2, 3

enum Bar {
  kKF = 0,        // [7] rank 0: slot group landed in both score ranks (1 arrival + TMA tx of both)
  kKE = 8,        // [7] score ranks: slot group free (commit from rank 0)
  kQRF = 16,      // rank 0: Q RoPE part landed in both score ranks (TMA tx of both)
  kQFree = 17,    // score ranks: both issuers' score MMAs of the segment finished (RoPE part may be replaced)
  kQF = 36,       // rank 0: both issuers' score MMAs of a segment finished (Q may be replaced)
  kQC = 37,       // rank 0: Q of the segment copied into tensor memory (commit from the first issuer)
  kSF = 38,       // [2] score ranks: scores ready (commit from rank 0)
  kSE = 40,       // [2] rank 0: scores read (one arrival per softmax warp of both ranks)
  kPFree = 42,    // [2] score ranks: the value rank is done with that P slot (commit from rank 2 after
                  //     PV; after a segment's last tile, an arrival from the epilogue that staged O there)
  kVF = 44,       // [4] value ranks: page slot landed (TMA tx)
  kVE = 48,       // [4] value ranks: page slot free (commit from rank 2)
  kVR = 52,       // [4] rank 2: page slot converted in both value ranks
  kPM = 56,       // [2] value ranks: P message landed (1 arrival + tx bytes)
  kPR = 58,       // [2] rank 2: O rescaled and P landed in both value ranks
  kPD = 60,       // [2] value ranks: PV of a tile of that parity finished (commit from rank 2)
  kOF = 62,       // value ranks: a segment's last PV finished (commit from rank 2)
  kOE = 63,       // rank 2: both value ranks' epilogues read O
  kMmaDone = 64,  // teardown
  kPsFull = 65,   // score ranks: the local P copy is written (one arrival per softmax warp)
  kPsFree = 66,   // score ranks: the bulk copy has read the local P copy
  kMmaDone2 = 67, // teardown (second issuer)
  kHand = 68,     // [2] rank 0: score-MMA issue token (tile parity): the issuer of tile g may start
                  //     once the issuer of tile g - 1 has issued two thirds of its MMAs
  kEpiD = 70,     // value ranks: the conversion warps' share of a segment epilogue is written
  kNumBars = 71
};
static_assert(kNumBars * 8 + 16 <= kBarBytes, "barrier block");
static_assert(kKGroups <= kKE - kKF && kKGroups <= kQRF - kKE, "slot-group barriers");

// Per segment the chunk ring carries pads, 16 Q halves (eight 16 KiB chunks,
// each two adjacent slots), then 9 K chunks per tile.  A segment starts on a
// group boundary u; q_pads(u) pads are inserted so that every Q chunk sits in
// two adjacent slots (none straddles the ring's end) and the tiles that
// follow start on a group boundary again.
__host__ __device__ constexpr uint32_t q_pads(uint32_t u) {
  return (u % kKSlots == 6u || u % kKSlots == 12u || u % kKSlots == 18u) ? 5u : 2u;
}
__host__ __device__ constexpr bool q_pads_ok() {
  for (uint32_t r = 0; r < kKSlots; r += kKGroup) {
    const uint32_t uq = r + q_pads(r);
    if ((uq + 16u) % kKGroup != 0u) return false;
    for (uint32_t i = 0; i < 8u; ++i)
      if ((uq + 2u * i) % kKSlots == kKSlots - 1u) return false;
  }
  return true;
}
static_assert(kKSlots % kKGroup == 0 && q_pads_ok(), "Q chunks stay contiguous; tiles stay group-aligned");

// kind::f16 instruction descriptors.  Scores: bf16 operands, M = 256, N = 128,
// B (the cached rows) K-major.  Values: fp16 or bf16 operands (A and B of
// one MMA always share a type), M = 256, N = 256, B (V) MN-major.
constexpr uint32_t kIdescQK = idesc_bf16(256, 128, 0);
template <bool kBf16PV>
__host__ __device__ constexpr uint32_t idesc_pv() {
  return (1u << 4) | ((kBf16PV ? 1u : 0u) << 7) | ((kBf16PV ? 1u : 0u) << 10) | (1u << 16) |
         ((256u >> 3) << 17) | ((256u >> 4) << 24);
}

// Position in an N-slot ring.
template <uint32_t N>
struct Ring {
  uint32_t idx = 0, phase = 0;
  __device__ void advance() {
    if (++idx == N) {
      idx = 0;
      phase ^= 1u;
    }
  }
};

// Bytes of one P message: the 16-bit P tile, the per-row rescale factor and,
// at the end of a segment, the per-row final scale.
__host__ __device__ constexpr uint32_t p_message_bytes(bool last) {
  return static_cast<uint32_t>(kPSlot + kHeads * 4 + (last ? kHeads * 4 : 0));
}

template <bool kBf16PV>
__global__ void __launch_bounds__(kThreads, 1)
mla_decode_mtp_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k3, const __grid_constant__ CUtensorMap tm_v2,
                      const __grid_constant__ CUtensorMap tm_out, const __grid_constant__ CUtensorMap tm_part) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t mis = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + mis;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t rank = cluster_ctarank();  // 0, 1: score pair; 2, 3: value pair
  const uint32_t tok = rank & 1u;           // the query token this CTA serves
  const bool score_rank = rank < 2;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int unit = blockIdx.x >> 2;

  // The set-up below overlaps the end of the plan kernel (a programmatic
  // dependency); nothing the plan writes is read before grid_dependency_wait.
  // The combine kernel may be scheduled at once: it waits for this grid too.
  grid_launch_dependents();
  if (mis > kAlignSlack) {  // never touch shared memory past the end of the allocation
    grid_dependency_wait();
    if (threadIdx.x == 0) atomicCAS(p.ws_hdr + kHdrStatus, 0, static_cast<int>(kStWorkspace));
    return;
  }

  auto kslot = [&](uint32_t i) -> uint32_t { return sbase + kOffStage + i * static_cast<uint32_t>(kPageChunk); };
  auto vslot = [&](uint32_t i) -> uint32_t { return sbase + kOffStage + i * static_cast<uint32_t>(kVPage); };
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * static_cast<uint32_t>(i); };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * kNumBars);
  // misc[0] = tensor-memory base, misc[1] = abort flag

  if (threadIdx.x == 0) {
    for (int i = 0; i < kKGroups; ++i) {
      mbar_init(bar(kKF + i), 1);
      mbar_init(bar(kKE + i), 1);
    }
    mbar_init(bar(kQRF), 1);
    mbar_init(bar(kQFree), 2);
    mbar_init(bar(kQC), 1);
    mbar_init(bar(kMmaDone2), 1);
    mbar_init(bar(kHand), 1);
    mbar_init(bar(kHand + 1), 1);
    for (int i = 0; i < kVSlots; ++i) {
      mbar_init(bar(kVF + i), 1);
      mbar_init(bar(kVE + i), 1);
      mbar_init(bar(kVR + i), kBf16PV ? 2 : 2 * (kConvThreads / 32));  // fp16: every conversion warp of both
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kSF + i), 1);
      mbar_init(bar(kSE + i), 2 * kSoftmaxWarps);
      mbar_init(bar(kPFree + i), 1);
      mbar_init(bar(kPM + i), 1);
      mbar_init(bar(kPR + i), 2);
      mbar_init(bar(kPD + i), 1);
    }
    mbar_init(bar(kQF), 2);
    mbar_init(bar(kOF), 1);
    mbar_init(bar(kOE), 2);
    mbar_init(bar(kMmaDone), 1);
    mbar_init(bar(kPsFull), kSoftmaxWarps);
    mbar_init(bar(kPsFree), 1);
    mbar_init(bar(kEpiD), 1);
    misc[1] = 0u;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(smem_u32(&misc[0]), kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(score_rank ? &tm_k3 : &tm_v2);
    if (!score_rank) {
      tma_prefetch_desc(&tm_out);
      tma_prefetch_desc(&tm_part);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // every CTA's barriers exist before any remote operation
  tc_fence_after();
  const uint32_t tmem = misc[0];
  grid_dependency_wait();  // the plan (unit ranges, request table) is complete
  // a set status word (a failed validation) leaves this step's outputs
  // unwritten: every role skips its work and the CTAs go straight to the
  // teardown (the plan and the check are complete here, and nothing else
  // writes the word before this grid's own waits could run out)
  const bool halt = p.ws_hdr[kHdrStatus] != 0;

  Ctl ctl;
  ctl.abort = &misc[1];
  ctl.n_remote = 0;
  for (uint32_t r = 0; r < 4; ++r)
    if (r != rank) ctl.abort_remote[ctl.n_remote++] = mapa(smem_u32(&misc[1]), r);
  ctl.status = p.ws_hdr + kHdrStatus;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const int U = p.num_units;

  // ======================================================= score-MMA issue (rank 0)
  // The chunk ring is consumed in "uses" of one 8 KiB slot: a K chunk, half
  // of a Q chunk (a Q chunk is two adjacent slots) or a pad.  Per segment:
  // 2 or 5 pads (so that Q starts on a slot = 2 mod 6: even, and its 16 uses
  // end on a group boundary), 16 Q uses, then 9 uses per tile; every tile is
  // three whole slot groups, owned by the issuer of that tile.  Issuer A
  // (even tiles, score buffer 0) also copies Q into tensor memory; issuer B
  // (odd tiles, score buffer 1) waits until that copy has completed.
  auto issue_scores = [&](bool is_a) {
    SegIter it(p, unit);
    Seg sg;
    uint32_t g = 0, nseg = 0, u = 0;
    bool ok = true;
    const uint32_t kf0 = bar(kKF), ke0 = bar(kKE), slot0 = sbase + kOffStage;
    const uint32_t own = is_a ? 0u : 1u;
    while (ok && it.next(sg)) {
      const uint32_t u_q = u + q_pads(u);
      const uint32_t u_t = u_q + 16u;  // first use of the segment's tiles (a group boundary)
      if (is_a) {
        if (nseg > 0 && !(ok = wait_bar<false>(bar(kQF), (nseg - 1u) & 1u, ctl))) break;
        // pads and Q may span seven slot groups, one more than the ring: wait,
        // copy and free chunk by chunk
        uint32_t gw = u / kKGroup, gf = u / kKGroup;  // next group to wait for / to free
        for (int i = 0; i < 8 && ok; ++i) {
          const uint32_t ue = u_q + 2u * i + 2u;  // uses [.., ue) are consumed by this copy
          for (; gw * kKGroup < ue && ok; ++gw) {
            ok = wait_bar<true>(kf0 + 8u * (gw % kKGroups), (gw / kKGroups) & 1u, ctl);
            tc_fence_after();
          }
          if (!ok) break;
          const uint64_t qd = smem_desc(slot0 + ((u_q + 2u * i) % kKSlots) * kPageChunk, 16u, 1024u);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tmem_cp_pair_128x256b(tmem + kColQ + 32u * i + 8u * kk, qd + static_cast<uint64_t>((32 * kk) >> 4));
          for (; (gf + 1) * kKGroup <= ue; ++gf) umma_commit_pair(ke0 + 8u * (gf % kKGroups), kScoreMask);
        }
        if (!ok) break;
        umma_commit_pair(bar(kQC), 1u << 0);
      } else {
        if (!(ok = wait_bar<false>(bar(kQC), nseg & 1u, ctl))) break;
        tc_fence_after();
      }
      u = u_t;
      if (!(ok = wait_bar<true>(bar(kQRF), nseg & 1u, ctl))) break;
      const uint64_t qr0 = smem_desc(sbase + kOffQr, 16u, 1024u);
      for (int j = sg.t0; j < sg.t1 && ok; ++j, ++g, u += kNumChunks) {
        const uint32_t sb = g & 1u, ph = (g >> 1) & 1u;
        if (sb != own) continue;
        if (!(ok = wait_bar<true>(bar(kSE + sb), ph ^ 1u, ctl))) break;
        if (!(ok = wait_bar<true>(kf0 + 8u * ((u / kKGroup) % kKGroups), ((u / kKGroup) / kKGroups) & 1u, ctl)))
          break;
        if (g > 0 && !(ok = wait_bar<false>(bar(kHand + ((g - 1u) & 1u)), ((g - 1u) >> 1) & 1u, ctl))) break;
        tc_fence_after();
        const uint32_t dS = tmem + kColS + 128u * sb;
        // K = 576 in 36 steps of 16, one 64-dim chunk per slot.  The next slot
        // group is probed (without blocking) one chunk into the current one:
        // a blocking wait, even on a completed barrier, stalls this thread for
        // ~150 cycles, in which the shallow MMA queue runs dry.
        uint32_t next_ready = 0;
#pragma unroll
        for (int c = 0; c < kNumChunks; ++c) {
          const uint32_t uc = u + c;
          const uint32_t G = uc / kKGroup;
          if (c == 6) mbar_arrive_relaxed(bar(kHand + sb));  // the other issuer may start its tile
          if (c > 0 && c % kKGroup == 0) {  // the next slot group (the first was waited for above)
            if (!next_ready && !(ok = wait_bar<true>(kf0 + 8u * (G % kKGroups), (G / kKGroups) & 1u, ctl))) break;
            tc_fence_after();
          }
          if (c % kKGroup == 1 && c + kKGroup < kNumChunks + 1)
            next_ready = mbar_test_wait_cluster(kf0 + 8u * ((G + 1u) % kKGroups), ((G + 1u) / kKGroups) & 1u);
          const uint64_t bd = smem_desc(slot0 + (uc % kKSlots) * kPageChunk, 16u, 1024u);
          if (c < 8) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_pair_ta(dS, tmem + kColQ + 32u * c + 8u * kk, bd + static_cast<uint64_t>((32 * kk) >> 4),
                           kIdescQK, (c | kk) != 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_pair_sa(dS, qr0 + static_cast<uint64_t>((32 * kk) >> 4),
                           bd + static_cast<uint64_t>((32 * kk) >> 4), kIdescQK, 1u);
          }
          if (c % kKGroup == kKGroup - 1) umma_commit_pair(ke0 + 8u * (G % kKGroups), kScoreMask);
        }
        if (!ok) break;
        umma_commit_pair(bar(kSF + sb), kScoreMask);
      }
      if (!ok) break;
      // this issuer's score MMAs of the segment: Q and the RoPE buffer may be replaced after both
      umma_commit_pair(bar(kQF), 1u << 0);
      umma_commit_pair(bar(kQFree), kScoreMask);
      ++nseg;
    }
    const uint32_t done = bar(is_a ? kMmaDone : kMmaDone2);
    umma_commit_pair(done, 1u << 0);  // every MMA this thread issued has finished
    drain_bar(done, 0);
  };

  // ======================================================= segment epilogue share
  // Warp w (0-15) of a value rank writes rows 32 (w % 4) .. +31 (its
  // tensor-memory lane quarter), columns 128 (w / 4) .. +127 of O times
  // `fin`: 32-row boxes of 64-byte rows (32 bf16 or 16 fp32 columns) staged
  // with the 64-byte swizzle in the warp's 2 KiB of P slot `pb` (free: PV has
  // finished with it, and the score rank refills it only after the epilogue)
  // and written by tensor stores, so both the shared-memory writes and the
  // global writes are full-width.
  auto epilogue_share = [&](int w, float fin, const Seg& sg, uint32_t pb) {
    const bool to_part = sg.slot >= 0;
    if (to_part && sg.slot >= 2 * U) return;  // the plan never uses more than 2 * (U - 1) slots
    const bool f32 = !to_part && p.out_fp32;  // partials are 16-bit (fp16, or bf16 with kBf16PV)
    const CUtensorMap* tm = to_part ? &tm_part : &tm_out;
    const long long orow = to_part ? static_cast<long long>(sg.slot) * 2 + tok : static_cast<long long>(sg.b) * 2 + tok;
    const int y = static_cast<int>(orow * kHeads) + 32 * (w & 3);
    const int x0 = 128 * (w >> 2);
    const uint32_t ul = static_cast<uint32_t>(lane);
    const uint32_t stg = sbase + kOffP + pb * kPSlot + static_cast<uint32_t>(w) * 2048u;
    const uint32_t srow = stg + ul * 64u, sw = (ul >> 1) & 3u;
    const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * (w & 3)) << 16) + kColO + static_cast<uint32_t>(x0);
    const int nbox = f32 ? 8 : 4, bw = f32 ? 16 : 32;
    // partial results stay in L2 for the combine kernel; final ones need not
    const uint64_t pol = to_part ? l2_policy_evict_last() : l2_policy_evict_first();
#pragma unroll 1
    for (int i = 0; i < nbox; ++i) {
      uint32_t v[16];
      if (f32) {
        uint32_t r[16];
        tmem_ld16(taddr + static_cast<uint32_t>(16 * i), r);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 16; ++c) v[c] = __float_as_uint(__uint_as_float(r[c]) * fin);
      } else {
        uint32_t r[32];
        tmem_ld32(taddr + static_cast<uint32_t>(32 * i), r);
        tmem_wait_ld();
        if (to_part && !kBf16PV) {
#pragma unroll
          for (int c = 0; c < 16; ++c)
            v[c] = pack_f16x2(__uint_as_float(r[2 * c]) * fin, __uint_as_float(r[2 * c + 1]) * fin);
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c)
            v[c] = pack_bf16x2(__uint_as_float(r[2 * c]) * fin, __uint_as_float(r[2 * c + 1]) * fin);
        }
      }
      if (i > 0) {  // the previous box's store has read the staging
        if (lane == 0) bulk_wait_read();
        __syncwarp();
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
        st_shared_v4(srow + ((static_cast<uint32_t>(k) ^ sw) << 4), v[4 * k], v[4 * k + 1], v[4 * k + 2],
                     v[4 * k + 3]);
      fence_proxy_async_smem();  // generic writes, read next by the tensor store
      __syncwarp();
      if (lane == 0) {
        tma_store_2d_hint(tm, stg, x0 + bw * i, y, pol);
        bulk_commit();
      }
    }
    if (lane == 0) bulk_wait_read();
    __syncwarp();
  };

  if (halt) {
    // nothing to do
  } else if (score_rank && warp < kSoftmaxWarps) {
    // ================================================= softmax (score ranks)
    // Warp (q4, cg): head rows 32 q4 .. +31 (its tensor-memory lane quarter),
    // key columns 32 cg .. +31 of the tile.  The four warps of a quarter
    // combine their row maxima through shared memory (named barrier 1 + q4).
    const int q4 = warp & 3, cg = warp >> 2;
    const int row = q4 * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const bool lead = cg == 0;  // the quarter's leading warp signals and writes the row scales
    // this thread's four 16-B pieces: half cg / 2 of the keys, pieces 4 (cg % 2) ..
    const uint32_t sProw = sbase + kOffPs + static_cast<uint32_t>(row >> 3) * kPGroupStride +
                           static_cast<uint32_t>(cg >> 1) * kPHalfStride + static_cast<uint32_t>(row & 7) * 128u;
    const uint32_t piece0 = static_cast<uint32_t>(cg & 1) * 4u;
    float* alpha_out = reinterpret_cast<float*>(smem + kOffAlphaS);
    float* fin_out = reinterpret_cast<float*>(smem + kOffFinS);
    const uint32_t rSE = mapa(bar(kSE), 0);
    float* xmax = reinterpret_cast<float*>(smem + kOffXchg);                   // [2 parity][4 cg][128]
    float* xsum = reinterpret_cast<float*>(smem + kOffXchg + 8 * kHeads * 4);  // [2 sum][4 cg][128]
    const int qbar = 1 + q4;
    SegIter it(p, unit);
    Seg sg;
    uint32_t g = 0;
    bool ok = true, stop = false;  // ok: this warp's waits so far; stop: the quarter leaves
    while (!stop && it.next(sg)) {
      const int L = max(p.cache_lens[sg.b], 0);
      const int vis = p.causal ? L - 1 + static_cast<int>(tok) : L;
      const long long bt_row = static_cast<long long>(sg.b) * 2 + tok;
      // zr: sum of the 16-bit weights the value product uses; it normalises O,
      // so O is a convex combination of value rows and a weight's rounding
      // error acts on (v_j - O) instead of v_j.  zx: sum of the fp32 weights,
      // for the LSE.  Each warp keeps the sums of its own 32 key columns.
      float m_used = NEG_INF, zr = 0.f, zx = 0.f;
      for (int j = sg.t0; j < sg.t1; ++j, ++g) {
        const uint32_t sb = g & 1u, ph = (g >> 1) & 1u;
        const bool last = (j == sg.t1 - 1);
        ok = ok && warp_wait(bar(kSF + sb), ph, ctl);
        float s[32];
        if (ok) {
          tc_fence_after();
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + kColS + 128u * sb + 32u * cg, r);
          tmem_wait_ld();
          tc_fence_before();
          // this warp has read its scores: the buffer's next tile may start
          // as soon as all 32 softmax warps of the pair have
          if (lane == 0) mbar_arrive_remote_relaxed(rSE + 8u * sb);
#pragma unroll
          for (int c = 0; c < 32; ++c) s[c] = __uint_as_float(r[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) s[c] = NEG_INF;
        }

        // ---- causal / length mask, then the row max over the quarter's warps
        const int nvalid = vis - (j * kTileRows + 32 * cg);
        if (nvalid < 32) {
#pragma unroll
          for (int c = 0; c < 32; ++c) s[c] = c < nvalid ? s[c] : NEG_INF;
        }
        {
          float m4[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
#pragma unroll
          for (int c = 0; c < 32; ++c) m4[c & 3] = fmaxf(m4[c & 3], s[c]);
          xmax[(sb * 4 + cg) * kHeads + row] = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        }
        if (!named_bar_all(qbar, 128, ok)) {
          stop = true;
          break;
        }
        const float* xm = xmax + sb * 4 * kHeads + row;
        const float mt = fmaxf(fmaxf(xm[0], xm[kHeads]), fmaxf(xm[2 * kHeads], xm[3 * kHeads])) * p.scale_log2;

        float alpha = 1.f;
        if (mt > m_used + kRescaleLog2) {
          alpha = (m_used == NEG_INF) ? 0.f : ex2_approx(m_used - mt);
          m_used = mt;
          zr *= alpha;
          zx *= alpha;
        }
        uint32_t pk[16];
        if (m_used == NEG_INF) {
#pragma unroll
          for (int c = 0; c < 16; ++c) pk[c] = 0u;
        } else {
          // the 16-bit weights are widened exactly and summed in fp32
          float zs[4] = {0.f, 0.f, 0.f, 0.f}, ze[4] = {0.f, 0.f, 0.f, 0.f};
          const float nm = -m_used;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float p0 = ex2_approx(fmaf(s[2 * c], p.scale_log2, nm));
            const float p1 = ex2_approx(fmaf(s[2 * c + 1], p.scale_log2, nm));
            pk[c] = kBf16PV ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
            zs[c & 3] = kBf16PV ? add_bf16x2_halves(zs[c & 3], pk[c]) : add_f16x2_halves(zs[c & 3], pk[c]);
            ze[c & 3] += p0 + p1;
          }
          zr += (zs[0] + zs[1]) + (zs[2] + zs[3]);
          zx += (ze[0] + ze[1]) + (ze[2] + ze[3]);
        }
        // ---- the local P copy: free once the previous tile's bulk copy read it
        if (g > 0) ok = ok && warp_wait(bar(kPsFree), (g - 1u) & 1u, ctl);
        if (ok) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            st_shared_v4(sProw + (((piece0 + static_cast<uint32_t>(k)) ^ (row & 7)) << 4), pk[4 * k],
                         pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
          if (lead) alpha_out[row] = alpha;
        }
        if (last) {  // ---- segment end: the quarter's partial sums -> final scale and LSE
          xsum[cg * kHeads + row] = zr;
          xsum[(4 + cg) * kHeads + row] = zx;
          if (!named_bar_all(qbar, 128, ok)) {
            stop = true;
            break;
          }
          if (lead) {
            const float zrt = (zr + xsum[kHeads + row]) + (xsum[2 * kHeads + row] + xsum[3 * kHeads + row]);
            const float zxt = (zx + xsum[5 * kHeads + row]) + (xsum[6 * kHeads + row] + xsum[7 * kHeads + row]);
            fin_out[row] = zrt > 0.f ? 1.f / zrt : 0.f;  // O_final = O_acc / zr
            const float lse = zxt > 0.f ? (m_used + log2f(zxt)) * 0.69314718055994531f : NEG_INF;
            if (sg.slot < 0) {
              p.lse[bt_row * kHeads + row] = lse;
            } else if (sg.slot < 2 * U) {  // the plan never uses more than 2 * (U - 1) slots
              p.part_lse[(static_cast<long long>(sg.slot) * 2 + tok) * kHeads + row] = lse;
            }
          }
        }
        if (ok) {
          fence_proxy_async_smem();  // generic writes above, read next by the bulk copy
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kPsFull));
        }
      }
    }
  } else if (score_rank && warp == kShipWarp) {
    // ================================================= P shipper (score ranks, one lane)
    if (lane == 0) {
      const uint32_t vrank = 2u + tok;
      const uint32_t rP = mapa(sbase + kOffP, vrank);
      const uint32_t rAlpha = mapa(sbase + kOffAlpha, vrank);
      const uint32_t rFin = mapa(sbase + kOffFin, vrank);
      const uint32_t rPM = mapa(bar(kPM), vrank);
      SegIter it(p, unit);
      Seg sg;
      uint32_t g = 0;
      bool ok = true;
      while (ok && it.next(sg)) {
        for (int j = sg.t0; j < sg.t1; ++j, ++g) {
          const uint32_t sb = g & 1u, ph = (g >> 1) & 1u;
          if (!(ok = wait_bar<false>(bar(kPsFull), g & 1u, ctl))) break;
          if (!(ok = wait_bar<false>(bar(kPFree + sb), ph ^ 1u, ctl))) break;  // PV is done with that slot
          const uint32_t mbar = rPM + 8u * sb;
          bulk_copy_s2c(rP + sb * kPSlot, sbase + kOffPs, static_cast<uint32_t>(kPSlot), mbar);
          bulk_copy_s2c(rAlpha + sb * kHeads * 4u, sbase + kOffAlphaS, kHeads * 4u, mbar);
          if (j == sg.t1 - 1) bulk_copy_s2c(rFin + sb * kHeads * 4u, sbase + kOffFinS, kHeads * 4u, mbar);
          bulk_commit();
          bulk_wait_read();
          mbar_arrive_relaxed(bar(kPsFree));  // execution token: the copy has read the local P
        }
      }
      bulk_wait_all();  // copies out of this CTA's memory are complete
    }
    __syncwarp();
  } else if (!score_rank && warp < 4) {
    // ================================================= O rescale + epilogue (value ranks)
    const int row = threadIdx.x;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const volatile float* alpha_s = reinterpret_cast<const volatile float*>(smem + kOffAlpha);
    const volatile float* fin_s = reinterpret_cast<const volatile float*>(smem + kOffFin);
    const uint32_t rPR = mapa(bar(kPR), 2);
    const uint32_t rOE = mapa(bar(kOE), 2);
    const uint32_t rPFree = mapa(bar(kPFree), tok);  // the score rank that ships this rank's P
    SegIter it(p, unit);
    Seg sg;
    uint32_t g = 0, nseg = 0;
    bool ok = true, stop = false;  // the four warps vote at every named barrier
    while (!stop && it.next(sg)) {
      float fin = 0.f;
      for (int j = sg.t0; j < sg.t1; ++j, ++g) {
        const uint32_t pb = g & 1u, ph = (g >> 1) & 1u;
        const bool last = (j == sg.t1 - 1);
        if (row == 0) mbar_arrive_expect_tx(bar(kPM + pb), p_message_bytes(last));
        ok = ok && warp_wait<true>(bar(kPM + pb), ph, ctl);
        const float alpha = ok ? alpha_s[pb * kHeads + row] : 1.f;
        if (last && ok) fin = fin_s[pb * kHeads + row];
        const bool resc = ok && (j != sg.t0) && alpha != 1.f;
        if (__any_sync(0xffffffffu, resc)) {  // tcgen05.ld/st are warp-collective
          // PV(g-1) finished: phase (g-1)/2 of the barrier of its parity (the
          // phase before it, PV(g-3), is known complete: P(g-1) was sent after it)
          const uint32_t gp = g - 1u;
          ok = warp_wait(bar(kPD + (gp & 1u)), (gp >> 1) & 1u, ctl);
        }
        if (__any_sync(0xffffffffu, resc) && ok) {
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
        fence_proxy_async_smem();  // P written by the bulk copy, read next by the tensor core
        tc_fence_before();
        if (!named_bar_all(5, 128, ok)) {
          stop = true;
          break;
        }
        // relaxed: what it hands over is P, whose landing this CTA observed on
        // its own barrier, and O rows whose rescale tcgen05.wait::st completed;
        // a release arrive would first wait for this thread's earlier memory
        // operations, a thousand cycles on the path of every tile
        if (row == 0) mbar_arrive_remote_relaxed(rPR + 8u * pb);

        if (last) {  // ---- segment epilogue: O * fin -> global, shared with the conversion warps
          ok = warp_wait(bar(kOF), nseg & 1u, ctl);
          if (!named_bar_all(5, 128, ok)) {
            stop = true;
            break;
          }
          tc_fence_after();
          epilogue_share(warp, fin, sg, pb);
          ok = warp_wait(bar(kEpiD), nseg & 1u, ctl);  // the other twelve warps' shares
          tc_fence_before();
          if (!named_bar_all(5, 128, ok)) {
            stop = true;
            break;
          }
          if (row == 0) {
            mbar_arrive_remote_relaxed(rOE);       // O read (tcgen05.wait::ld completed in all 16 warps)
            mbar_arrive_remote(rPFree + 8u * pb);  // the staging (this P slot) is free again
          }
        }
      }
      ++nseg;
    }
    if (lane == 0) bulk_wait_all();  // the output stores have completed
  } else if (warp == kMmaWarp || warp == kMma2Warp) {
    // ================================================= MMA issue (rank 0: two threads, rank 2: one)
    if (lane == 0 && rank == 0) {
      issue_scores(warp == kMmaWarp);
    } else if (lane == 0 && rank == 2 && warp == kMmaWarp) {
      SegIter it(p, unit);
      Seg sg;
      Ring<kVSlots> rv;
      uint32_t g = 0, nseg = 0;
      bool ok = true;
      constexpr uint32_t kIdescPV = idesc_pv<kBf16PV>();
      while (ok && it.next(sg)) {
        for (int j = sg.t0; j < sg.t1 && ok; ++j, ++g) {
          const uint32_t pb = g & 1u, ph = (g >> 1) & 1u;
          const bool first = (j == sg.t0);
          if (!(ok = wait_bar<true>(bar(kPR + pb), ph, ctl))) break;
          if (first && !(ok = wait_bar<true>(bar(kOE), (nseg & 1u) ^ 1u, ctl))) break;
          const uint64_t ad0 = smem_desc(sbase + kOffP + pb * kPSlot, 16u, static_cast<uint32_t>(kPGroupStride));
          // the tile's two pages, 64 keys each (K = 4 x 16 per page)
#pragma unroll 1
          for (int e = 0; e < 2; ++e, rv.advance()) {
            if (!(ok = wait_bar<true>(bar(kVR + rv.idx), rv.phase, ctl))) break;
            tc_fence_after();
            const uint64_t bd0 = smem_desc(vslot(rv.idx), static_cast<uint32_t>(kPageChunk), 1024u);  // MN-major
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
              for (int h = 0; h < 2; ++h)
                umma_pair_sa(tmem + kColO + 256u * h,
                             ad0 + static_cast<uint64_t>((e * kPHalfStride + kk * 32) >> 4),
                             bd0 + static_cast<uint64_t>((h * 2 * kPageChunk + 2048 * kk) >> 4), kIdescPV,
                             (first && e == 0 && kk == 0) ? 0u : 1u);
            }
            umma_commit_pair(bar(kVE + rv.idx), kValueMask);
          }
          if (!ok) break;
          // the score ranks may reuse this P slot (after a segment's last tile the
          // epilogue stages O there and frees it)
          if (j != sg.t1 - 1) umma_commit_pair(bar(kPFree + pb), kScoreMask);
          umma_commit_pair(bar(kPD + pb), kValueMask);
          if (j == sg.t1 - 1) umma_commit_pair(bar(kOF), kValueMask);
        }
        ++nseg;
      }
      umma_commit_pair(bar(kMmaDone), 1u << 2);
      drain_bar(bar(kMmaDone), 0);
    }
    __syncwarp();
  } else if (warp == kTmaWarp) {
    // ================================================= TMA producers (whole warp; lane 0 issues)
    // Page ids are read 32 tiles at a time with one coalesced load; a page
    // past the cache end or outside the pool reads the TMA fill value (zeros).
    SegIter it(p, unit);
    Seg sg;
    uint32_t issued = 0;
    bool ok = true;
    if (score_rank) {
      // Both score ranks fill their own chunk slots; every copy completes on
      // rank 0's barriers, which rank 0 arms with the bytes of both.  The use
      // sequence is the issuers': per segment q_pads() pads, 16 Q halves,
      // then 9 K chunks per tile.
      const uint32_t rKF = mapa(bar(kKF), 0);
      const uint32_t rQRF = mapa(bar(kQRF), 0);
      uint32_t u = 0, nseg = 0;
      // claim the next slot: wait for its group to be free at the group's
      // first use, add its bytes (both ranks) to the group's landing barrier,
      // and arrive once at the group's last use.  Relaxed forms: the
      // producer writes none of the data, and release semantics make each
      // barrier operation wait for the thread's earlier memory operations.
      auto claim = [&](uint32_t bytes) -> bool {
        const uint32_t sl = u % kKSlots, grp = sl / kKGroup;
        if (sl % kKGroup == 0 && !warp_wait(bar(kKE + grp), ((u / kKSlots) & 1u) ^ 1u, ctl)) return false;
        if (lane == 0 && tok == 0) {
          if (sl % kKGroup == kKGroup - 1) mbar_arrive_expect_tx_relaxed(bar(kKF + grp), 2u * bytes);
          else if (bytes) mbar_expect_tx_relaxed(bar(kKF + grp), 2u * bytes);
        }
        return true;
      };
      while (ok && it.next(sg)) {
        const int L = max(p.cache_lens[sg.b], 0);
        const int qy = (sg.b * 2 + static_cast<int>(tok)) * kHeads;
        for (uint32_t npad = q_pads(u); npad > 0 && ok; --npad) {  // pads
          if (!(ok = claim(0))) break;
          ++u;
        }
        for (int i = 0; i < 8 && ok; ++i) {
          for (int h = 0; h < 2; ++h) {
            if (!(ok = claim(kPageChunk))) break;
            if (lane == 0)
              tma_load_2d_pair(kslot(u % kKSlots), &tm_q, i * kChunk, qy + h * kPage,
                               rKF + 8u * ((u % kKSlots) / kKGroup));
            ++u;
          }
        }
        if (!ok) break;
        // RoPE part of Q (not in the ring) once the previous segment's score MMAs are done with it
        if (nseg >= 1 && !(ok = warp_wait(bar(kQFree), (nseg - 1u) & 1u, ctl))) break;
        if (lane == 0) {
          if (tok == 0) mbar_arrive_expect_tx_relaxed(bar(kQRF), 2u * kQChunk);
          for (int h = 0; h < 2; ++h)
            tma_load_2d_pair(sbase + kOffQr + h * kPageChunk, &tm_q, 8 * kChunk, qy + h * kPage, rQRF);
        }
        const int* bt_row = p.block_table + static_cast<long long>(sg.b) * p.bt_stride;
        const int npages = (L + kPage - 1) / kPage;
        for (int jb = sg.t0; jb < sg.t1 && ok; jb += 32) {
          const int cnt = min(32, sg.t1 - jb);
          int my_page = -1;
          const int pi = 2 * (jb + lane) + static_cast<int>(tok);
          if (lane < cnt && pi < npages && pi < p.bt_stride) {
            const int pg = bt_row[pi];
            my_page = (pg >= 0 && pg < p.num_pages) ? pg : -1;
          }
          for (int jj = 0; jj < cnt && ok; ++jj) {
            const int page = __shfl_sync(0xffffffffu, my_page, jj);
            const int y = page >= 0 ? page * kPage : static_cast<int>(p.num_pages) * kPage;
            // a tile is three whole slot groups: one 3-chunk load per group
            for (int c = 0; c < kNumChunks; c += kKGroup) {
              const uint32_t sl = u % kKSlots, grp = sl / kKGroup;
              if (!(ok = warp_wait(bar(kKE + grp), ((u / kKSlots) & 1u) ^ 1u, ctl))) break;
              if (lane == 0) {
                if (tok == 0) mbar_arrive_expect_tx_relaxed(bar(kKF + grp), 2u * kKGroup * kPageChunk);
                tma_load_3d_pair(kslot(sl), &tm_k3, 0, y, c, rKF + 8u * grp);
              }
              u += kKGroup;
            }
          }
        }
        ++nseg;
      }
      issued = u;
      if (!ok && lane == 0) {  // let copies in flight land before the CTA goes away
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < kDrainNs / 8) {
        }
      }
    } else {
      // Value ranks: per page, this rank's 256 value dims, the page's last
      // read in this step (the score rank read it just before): evict first.
      // At the start the score ranks' TMA units are the bottleneck (each
      // holds a limited number of bytes in flight while its Q streams in
      // from HBM): this rank pulls its token's Q and the first two pages of
      // that token into L2 meanwhile.
      const uint64_t pol_v = l2_policy_evict_first();
      if (lane == 0) {
        SegIter it0(p, unit);
        Seg s0;
        if (it0.next(s0)) {
          const long long qrow = (static_cast<long long>(s0.b) * 2 + tok) * kHeads;
          for (int h = 0; h < 2; ++h) bulk_prefetch_l2(p.q + (qrow + h * kPage) * kDqk, kPage * kDqk * 2);
          const int nl = max(p.cache_lens[s0.b], 0);
          const int np = (nl + kPage - 1) / kPage;
          const int* row = p.block_table + static_cast<long long>(s0.b) * p.bt_stride;
          for (int t = s0.t0; t < s0.t1 && t < s0.t0 + 2; ++t) {
            const int pi = 2 * t + static_cast<int>(tok);
            if (pi >= np || pi >= p.bt_stride) break;
            const int pg = row[pi];
            if (pg >= 0 && pg < p.num_pages)
              bulk_prefetch_l2(p.kv + static_cast<long long>(pg) * kPage * kDqk, kPage * kDqk * 2);
          }
        }
      }
      // (fp16 variant: the conversion warps load the value dims themselves)
      Ring<kVSlots> rv;
      while (kBf16PV && ok && it.next(sg)) {
        const int L = max(p.cache_lens[sg.b], 0);
        const int* bt_row = p.block_table + static_cast<long long>(sg.b) * p.bt_stride;
        const int npages = (L + kPage - 1) / kPage;
        for (int jb = sg.t0; jb < sg.t1 && ok; jb += 32) {
          const int cnt = min(32, sg.t1 - jb);
          int pg2[2] = {-1, -1};
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int pi = 2 * (jb + lane) + e;
            if (lane < cnt && pi < npages && pi < p.bt_stride) {
              const int pg = bt_row[pi];
              pg2[e] = (pg >= 0 && pg < p.num_pages) ? pg : -1;
            }
          }
          for (int jj = 0; jj < cnt && ok; ++jj) {
#pragma unroll 1
            for (int e = 0; e < 2; ++e, rv.advance()) {
              const int page = __shfl_sync(0xffffffffu, e ? pg2[1] : pg2[0], jj);
              if (!(ok = warp_wait(bar(kVE + rv.idx), rv.phase ^ 1u, ctl))) break;
              if (lane == 0) {
                const int y = page >= 0 ? page * kPage : static_cast<int>(p.num_pages) * kPage;
                mbar_arrive_expect_tx_relaxed(bar(kVF + rv.idx), kVPage);
                // chunks 2 tok, 2 tok + 1 and 4 + 2 tok, 5 + 2 tok: two loads of two chunks
#pragma unroll
                for (int h = 0; h < 2; ++h)
                  tma_load_3d_hint(vslot(rv.idx) + 2 * h * kPageChunk, &tm_v2, 0, y,
                                   4 * h + 2 * static_cast<int>(tok), bar(kVF + rv.idx), pol_v);
              }
              ++issued;
            }
          }
        }
      }
      if (!ok && lane == 0) {
        for (uint32_t k = 0; k < static_cast<uint32_t>(kVSlots) && k < issued; ++k) {
          const uint32_t t = issued - 1 - k;
          drain_bar(bar(kVF + t % kVSlots), (t / kVSlots) & 1u);
        }
      }
    }
  } else if (!score_rank && warp < kMmaWarp && !kBf16PV) {
    // ================================================= V loads + fp16 conversion (value ranks, warps 4-15)
    // fp16 variant.  Each page of this rank's value dims (64 rows x the
    // 128-dim halves [128 tok, +128) and [256 + 128 tok, +128)) is read from
    // global memory into registers (an L2 hit: the score rank has just
    // loaded the page), converted to fp16 and stored in the slot's 128B-
    // swizzled layout, the one the tensor loads give the bf16 variant.  Warp
    // w (0-11) owns rows w, w + 12, .. of a page; lanes 0-15 the first half
    // of a row, lanes 16-31 the second, 16 B each.  Staging through registers
    // instead of converting a landed tile in place halves this SM's shared-
    // memory traffic for V and frees a slot as soon as its value product is
    // done: the next page is loaded while the warps wait for the next free
    // slot.  Rows past the cache end (and pages outside the pool) are stored
    // as zeros, so whatever lies there cannot reach O.
    const int ptid = threadIdx.x - 128;
    const int lw = ptid >> 5;
    const int hs = lane >> 4, kp = lane & 15;
    const int gcol = 64 * (4 * hs + 2 * static_cast<int>(tok) + (kp >> 3)) + 8 * (kp & 7);
    const uint32_t scol = static_cast<uint32_t>((2 * hs + (kp >> 3)) * kPageChunk);
    const uint32_t spc = static_cast<uint32_t>(kp & 7);
    constexpr int kRowsPerThread = (kPage + 11) / 12;  // 6: rows lw + 12 i
    const volatile float* fin_s = reinterpret_cast<const volatile float*>(smem + kOffFin);
    // kVDepth pages of loads in flight per thread (registers), so that a
    // page's load latency spans several pages' turns
    uint4 v[kVDepth][kRowsPerThread];
    // Page ids of the segment, 32 at a time and one batch ahead: lane j holds
    // the pool page of page ids_base + j (-1 past the cache end or outside the
    // pool).  Reading the block-table entry next to each page's loads would
    // put an L2 round trip (the entry does not stay in the small L1 that the
    // value stream passes through) in front of every page.
    const int* bt_row = nullptr;
    int L = 0, ids_base = 0, ids_cur = -1, ids_next = -1;
    auto fetch_ids = [&](int base) {
      const int pi = base + lane;
      int page = -1;
      if (pi < (L + kPage - 1) / kPage && pi < p.bt_stride) {
        const int pg = __ldg(bt_row + pi);
        page = (pg >= 0 && pg < p.num_pages) ? pg : -1;
      }
      return page;
    };
    // page pi of the current segment's request into buffer dst; rows >= L -
    // 64 pi are zeros.  Called by whole warps with pi increasing by one.
    auto load_page = [&](uint4 (&dst)[kRowsPerThread], int pi) {
      if (pi >= ids_base + 32) {
        ids_base += 32;
        ids_cur = ids_next;
        ids_next = fetch_ids(ids_base + 32);
      }
      const int page = __shfl_sync(0xffffffffu, ids_cur, pi - ids_base);
      const int rows = L - pi * kPage;
      const uint16_t* src = p.kv + static_cast<long long>(page >= 0 ? page : 0) * (kPage * kDqk) + gcol;
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        const int r = lw + 12 * i;
        dst[i] = (page >= 0 && r < kPage && r < rows) ? ld_global_nc_v4(src + r * kDqk) : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    const uint32_t rVR = mapa(bar(kVR), 2);
    SegIter it(p, unit);
    Seg sg;
    Ring<kVSlots> rv;
    uint32_t g = 0, nseg = 0;
    // this warp's waits so far; the twelve warps vote at each segment's
    // epilogue barrier, so a warp whose wait failed skips the rest of the
    // segment's pages and they all leave there together
    bool wok = true;
    while (it.next(sg)) {
      L = max(p.cache_lens[sg.b], 0);
      bt_row = p.block_table + static_cast<long long>(sg.b) * p.bt_stride;
      const int p0 = 2 * sg.t0, np = 2 * (sg.t1 - sg.t0);  // this segment's pages: p0 .. p0 + np - 1
      ids_base = p0;
      ids_cur = fetch_ids(p0);
      ids_next = fetch_ids(p0 + 32);
#pragma unroll
      for (int d = 0; d < kVDepth; ++d)
        if (wok && d < np) load_page(v[d], p0 + d);
      for (int q0 = 0; q0 < np; q0 += kVDepth) {
#pragma unroll
        for (int d = 0; d < kVDepth; ++d) {
          const int q = q0 + d;
          if (q >= np) break;
          wok = wok && warp_wait(bar(kVE + rv.idx), rv.phase ^ 1u, ctl);  // PV is done with the slot
          if (wok) {
            const uint32_t stg = vslot(rv.idx) + scol;
#pragma unroll
            for (int i = 0; i < kRowsPerThread; ++i) {
              const int r = lw + 12 * i;
              if (r < kPage)
                st_shared_v4(stg + static_cast<uint32_t>(r) * 128u + ((spc ^ static_cast<uint32_t>(r & 7)) << 4),
                             bf16x2_to_f16x2(v[d][i].x), bf16x2_to_f16x2(v[d][i].y),
                             bf16x2_to_f16x2(v[d][i].z), bf16x2_to_f16x2(v[d][i].w));
            }
            fence_proxy_async_smem();  // generic writes, read next by the tensor core
            __syncwarp();
            // Each warp announces its own rows to rank 2 (release, cumulative
            // over the warp's stores), before its loads of the next page.  One
            // announcer per rank after a group barrier put that barrier and
            // the announcer's release on every page's path.
            if (lane == 0) mbar_arrive_remote_cta(rVR + 8u * rv.idx);
          }
          rv.advance();
          // the segment's page kVDepth ahead goes into the buffer just stored
          if (wok && q + kVDepth < np) load_page(v[d], p0 + q + kVDepth);
        }
      }
      g += static_cast<uint32_t>(sg.t1 - sg.t0);
      {  // ---- this group's share of the segment epilogue
        const uint32_t pb = (g - 1u) & 1u;  // the segment's last tile
        // O complete; the last P message (with the final scales) landed
        bool ok = wok && warp_wait(bar(kOF), nseg & 1u, ctl) && warp_wait(bar(kPM + pb), ((g - 1u) >> 1) & 1u, ctl);
        if (!named_bar_all(6, kConvThreads, ok)) break;
        tc_fence_after();
        epilogue_share(warp, fin_s[pb * kHeads + 32 * (warp & 3) + lane], sg, pb);
        tc_fence_before();
        named_bar_sync(6, kConvThreads);
        if (ptid == 0) mbar_arrive(bar(kEpiD));
      }
      ++nseg;
    }
    if (lane == 0) bulk_wait_all();  // the output stores have completed
  } else if (!score_rank && warp < kMmaWarp) {
    // ================================================= V tail zeroing (value ranks, warps 4-15, bf16 variant)
    const int ptid = threadIdx.x - 128;
    const uint32_t rVR = mapa(bar(kVR), 2);
    constexpr int kPieces = kVPage / 16;  // 2048 pieces of 16 B
    const volatile float* fin_s = reinterpret_cast<const volatile float*>(smem + kOffFin);
    SegIter it(p, unit);
    Seg sg;
    Ring<kVSlots> rv;
    uint32_t g = 0, nseg = 0;
    bool stop = false;  // the twelve warps vote at every named barrier
    while (!stop && it.next(sg)) {
      const int L = max(p.cache_lens[sg.b], 0);
      for (int j = sg.t0; j < sg.t1 && !stop; ++j, ++g) {
        for (int e = 0; e < 2; ++e, rv.advance()) {
          const bool ok = warp_wait(bar(kVF + rv.idx), rv.phase, ctl);
          if (!named_bar_all(6, kConvThreads, ok)) {
            stop = true;
            break;
          }
          const uint32_t stg = vslot(rv.idx);
          const int r_end = L - j * kTileRows - e * kPage;  // rows >= r_end lie past the cache end: zero them
          if (r_end < kPage) {
            for (int piece = ptid; piece < kPieces; piece += kConvThreads) {
              const int r = (piece & 511) >> 3;  // the swizzle only permutes pieces within a row
              if (r >= r_end) st_shared_zero16(stg + 16u * piece);
            }
          }
          fence_proxy_async_smem();
          named_bar_sync(6, kConvThreads);
          if (ptid == 0) mbar_arrive_remote_cta(rVR + 8u * rv.idx);
        }
        if (!stop && j == sg.t1 - 1) {  // ---- this group's share of the segment epilogue
          const uint32_t pb = g & 1u;
          // O complete; the last P message (with the final scales) landed
          bool ok = warp_wait(bar(kOF), nseg & 1u, ctl) && warp_wait(bar(kPM + pb), (g >> 1) & 1u, ctl);
          if (!named_bar_all(6, kConvThreads, ok)) {
            stop = true;
            break;
          }
          tc_fence_after();
          epilogue_share(warp, fin_s[pb * kHeads + 32 * (warp & 3) + lane], sg, pb);
          tc_fence_before();
          named_bar_sync(6, kConvThreads);
          if (ptid == 0) mbar_arrive(bar(kEpiD));
        }
      }
      ++nseg;
    }
    if (lane == 0) bulk_wait_all();  // the output stores have completed
  }

  // ======================================================= teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA touches another's shared memory after this
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// Launch configuration; `dependent`: may start while the previous kernel on
// the stream (the plan) finishes (programmatic dependent launch).
template <bool kBf16PV>
void cluster_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int num_clusters, cudaStream_t stream,
                    bool dependent) {
  cfg = cudaLaunchConfig_t{};
  cfg.gridDim = dim3(4 * num_clusters, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 4;  // two SM pairs
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 2 : 1;
}

}  // namespace mtp

// ------------------------------------------------------------------ host side
cudaError_t mtp_set_attrs() {
  cudaError_t e = cudaFuncSetAttribute(mtp::mla_decode_mtp_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, mtp::kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mtp::mla_decode_mtp_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              mtp::kSmemBytes);
}

// Co-resident 4-CTA clusters of the two-token kernel on the current device.
cudaError_t mtp_max_clusters(int* n, int num_clusters_hint) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  mtp::cluster_config<false>(cfg, attr, num_clusters_hint, nullptr, false);
  return cudaOccupancyMaxActiveClusters(n, mtp::mla_decode_mtp_kernel<false>, &cfg);
}

cudaError_t mtp_launch(bool bf16_pv, int num_clusters, cudaStream_t stream, const DecodeParams& p,
                       const CUtensorMap& tm_q, const CUtensorMap& tm_k3, const CUtensorMap& tm_v2,
                       const CUtensorMap& tm_out, const CUtensorMap& tm_part) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  mtp::cluster_config<false>(cfg, attr, num_clusters, stream, true);
  return bf16_pv
      ? cudaLaunchKernelEx(&cfg, mtp::mla_decode_mtp_kernel<true>, p, tm_q, tm_k3, tm_v2, tm_out, tm_part)
      : cudaLaunchKernelEx(&cfg, mtp::mla_decode_mtp_kernel<false>, p, tm_q, tm_k3, tm_v2, tm_out, tm_part);
}

}  // namespace mla
