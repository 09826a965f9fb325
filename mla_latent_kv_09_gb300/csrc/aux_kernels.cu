// aux_kernels.cu — the split-KV planner, the LSE combine and the input
// validator of the MLA decode library (sm_103a).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "plan.cuh"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace mla {

// ------------------------------------------------------------------ plan
constexpr int kPlanSmemReqs = 4096;  // requests whose cost prefix the plan keeps in shared memory
// Block-wide inclusive scan of one int per thread (up to 1024 threads).
__device__ int block_inclusive_scan(int v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) s_warp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (blockDim.x >> 5) ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    s_warp[lane] = w;  // inclusive per-warp totals
  }
  __syncthreads();
  const int res = v + (warp > 0 ? s_warp[warp - 1] : 0);
  total = s_warp[(blockDim.x >> 5) - 1];
  __syncthreads();
  return res;
}

// One CTA (128 threads up to 128 requests, else 1024).  Step 1: tiles and
// cost prefix per request.
// Step 2: split count and first partial slot per request.  Step 3: the
// (request, tile) range of every unit, by binary search over the cost
// prefixes (kept in shared memory when they fit: the searches are chains of
// dependent reads).  Also resets the status word.
__global__ void __launch_bounds__(1024) mla_plan_kernel(const int* __restrict__ lens, int B, int topk,
                                                        int tile_rows, int U, int* hdr, int* unit_meta,
                                                        int* req_meta, int slots_cap) {
  __shared__ int s_warp[32];
  __shared__ int s_prefix[kPlanSmemReqs];  // exclusive cost prefix per request
  __shared__ int s_tiles[kPlanSmemReqs];   // tiles per request
  grid_launch_dependents();  // the decode kernel may set up now; it waits for this grid before reading the plan
  // Up to kPlanSmemReqs requests the table is built in shared memory and each
  // request's row is written once; beyond, the global rows hold the pass-one
  // values in between.
  const bool in_smem = B <= kPlanSmemReqs;
  int carry = 0, tot = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    const int n = b < B ? plan_tiles(max(lens[b], 0), topk, tile_rows) : 0;
    const int c = plan_cost(n);
    const int incl = block_inclusive_scan(c, s_warp, tot);
    if (b < B) {
      if (in_smem) {
        s_prefix[b] = carry + incl - c;
        s_tiles[b] = n;
      } else {
        req_meta[4 * b + 0] = n;
        req_meta[4 * b + 3] = carry + incl - c;
      }
    }
    carry += tot;
  }
  const int total = carry;
  const int W = plan_width(total, U);
  __syncthreads();
  carry = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int n = 0, pre = 0, ns = 0;
    if (b < B) {
      n = in_smem ? s_tiles[b] : req_meta[4 * b + 0];
      pre = in_smem ? s_prefix[b] : req_meta[4 * b + 3];
      ns = plan_n_splits(pre, n, W, U);
    }
    const int need = ns > 1 ? ns : 0;
    const int incl = block_inclusive_scan(need, s_warp, tot);
    if (b < B) reinterpret_cast<int4*>(req_meta)[b] = make_int4(n, ns, carry + incl - need, pre);
    carry += tot;
  }
  __syncthreads();
  auto prefix = [&](int b) { return in_smem ? s_prefix[b] : req_meta[4 * b + 3]; };
  for (int u = threadIdx.x; u < U; u += blockDim.x) {
    const UnitInfo ui = plan_unit(u, W, total, B, prefix);
    int* m = unit_meta + 5 * u;
    m[0] = ui.begin_req; m[1] = ui.begin_tile; m[2] = ui.end_req; m[3] = ui.end_tile;
    m[4] = ui.first_split;
  }
  if (threadIdx.x == 0) {
    hdr[kHdrStatus] = carry > slots_cap ? static_cast<int>(kStWorkspace) : 0;
    hdr[kHdrUnits] = U;
    hdr[kHdrWidth] = W;
    hdr[kHdrTotal] = total;
    hdr[kHdrSlots] = carry;
  }
}

// ------------------------------------------------------------------ combine
// Grid (min(B * s_q, 76), 128 / 8), one wave of 256-thread blocks on 152
// SMs: block x takes (request, token) rows x, x + gridDim.x, ..; warp w of
// a block merges head blockIdx.y * 8 + w.
// Requests with one split were finished by the decode kernel; requests with
// no tiles get O = 0, LSE = -inf.
__global__ void __launch_bounds__(256) mla_combine_kernel(const int* __restrict__ hdr,
                                                          const int* __restrict__ req_meta,
                                                          const float* __restrict__ part_lse,
                                                          const uint16_t* __restrict__ part_o, int part_bf16,
                                                          int s_q, int out_fp32, void* out, float* lse, int n_bt) {
  grid_launch_dependents();  // a kernel launched after this one may set up (it waits for this grid)
  grid_dependency_wait();    // the decode kernel has finished (programmatic dependent launch)
  if (hdr[kHdrStatus] != 0) return;  // a failed check or wait: the step's outputs stay unwritten
  for (int bt = blockIdx.x; bt < n_bt; bt += gridDim.x) {
    const int b = bt / s_q, t = bt - b * s_q;
    const int ns = req_meta[4 * b + 1];
    if (ns == 1) continue;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y * 8 + warp;
    const long long orow = (static_cast<long long>(bt) * kHeads + h) * kDv;
    float acc[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) acc[k] = 0.f;
    float LSE = -INFINITY;
    if (ns > 1) {
      // Lane s (< 32) holds split s's LSE: one round trip for the LSEs, shuffles
      // for max, sum and weights, then the partial rows of two splits per
      // batch (eight 16-byte loads in flight per lane).
      const int slot0 = req_meta[4 * b + 2];
      auto lse_of = [&](int s) { return part_lse[(static_cast<long long>(slot0 + s) * s_q + t) * kHeads + h]; };
      const float lse_l = lane < ns ? lse_of(lane) : -INFINITY;
      float m = lse_l;
      for (int s = lane + 32; s < ns; s += 32) m = fmaxf(m, lse_of(s));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (m != -INFINITY) {
        float sum = lane < ns ? expf(lse_l - m) : 0.f;
        for (int s = lane + 32; s < ns; s += 32) sum += expf(lse_of(s) - m);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        LSE = m + logf(sum);
        const float w_l = lane < ns ? expf(lse_l - LSE) : 0.f;
        // partial rows are 16-bit (fp16, or bf16 with MLA_FLAG_BF16_PV): lane
        // reads dims {4*lane + 128*k .. +3} as one 8-byte piece per k
        auto row = [&](int s) {
          return reinterpret_cast<const uint2*>(
                     part_o + ((static_cast<long long>(slot0 + s) * s_q + t) * kHeads + h) * kDv) + lane;
        };
        auto widen = [&](uint2 u) {
          float4 f;
          if (part_bf16) {
            f.x = __uint_as_float(u.x << 16); f.y = __uint_as_float(u.x & 0xffff0000u);
            f.z = __uint_as_float(u.y << 16); f.w = __uint_as_float(u.y & 0xffff0000u);
          } else {
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
            const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
            f = make_float4(a.x, a.y, b.x, b.y);
          }
          return f;
        };
        auto add = [&](float w, const float4 (&v)[4]) {
          if (w == 0.f) return;  // an empty split adds nothing
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            acc[4 * k + 0] += w * v[k].x; acc[4 * k + 1] += w * v[k].y;
            acc[4 * k + 2] += w * v[k].z; acc[4 * k + 3] += w * v[k].w;
          }
        };
        const int n32 = ns < 32 ? ns : 32;
        int s = 0;
        for (; s + 2 <= n32; s += 2) {
          const uint2* r0 = row(s);
          const uint2* r1 = row(s + 1);
          uint2 u0[4], u1[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            u0[k] = r0[32 * k];
            u1[k] = r1[32 * k];
          }
          float4 v0[4], v1[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            v0[k] = widen(u0[k]);
            v1[k] = widen(u1[k]);
          }
          add(__shfl_sync(0xffffffffu, w_l, s), v0);
          add(__shfl_sync(0xffffffffu, w_l, s + 1), v1);
        }
        for (; s < ns; ++s) {  // the odd split, and splits past 32
          const float w = s < 32 ? __shfl_sync(0xffffffffu, w_l, s) : expf(lse_of(s) - LSE);
          const uint2* r0 = row(s);
          float4 v0[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) v0[k] = widen(r0[32 * k]);
          add(w, v0);
        }
      }
    }
    // lane covers dims {4*lane + 128*k .. +3}, k = 0..3 (coalesced 16-byte pieces)
    if (out_fp32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + orow) + lane;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        dst[32 * k] = make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
    } else {
      uint2* dst = reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + orow) + lane;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t lo, hi;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(acc[4 * k + 1]), "f"(acc[4 * k]));
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(acc[4 * k + 3]), "f"(acc[4 * k + 2]));
        dst[32 * k] = make_uint2(lo, hi);
      }
    }
    if (lane == 0) lse[static_cast<long long>(bt) * kHeads + h] = LSE;
  }
}

// ------------------------------------------------------------------ validate
// Checks lengths, the block-table entries the step will read and the top-k
// indices, and (check_range) that every value dim the step reads is finite
// and converts to fp16 without overflow: check_range 1, a bf16 cache, |v| <
// 65536 as a bf16 pattern below 0x4780; check_range 2, an FP8 cache (656-byte
// rows), no NaN code, no scale byte 255, and |code| * scale < 65536 (every
// such value is at most 61440); records the first problem found in the
// status word.  One
// CTA per request (grid-strided); reading the value dims of every visible row
// makes this a full pass over the visible cache.
__global__ void mla_validate_kernel(const int* __restrict__ lens, const int* __restrict__ bt,
                                    long long bt_stride, long long num_pages, int B, int s_q,
                                    const int* __restrict__ topk_idx, int topk, const uint16_t* __restrict__ kv,
                                    int check_range, int* status) {
  __shared__ int s_bad;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  // value dims 0..511 of pool row `row`: one warp, 16 B per lane, 2 rounds
  auto row_in_range = [&](long long row) {
    if (check_range == 2) {  // FP8 row: lane l holds codes 16 l .. 16 l + 15 (scale group l / 8)
      const uint8_t* r8 = reinterpret_cast<const uint8_t*>(kv) + row * 656;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(r8) + lane);
      const uint32_t eb = __ldg(r8 + 512 + (lane >> 3));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      bool ok = eb != 255u;
      float mx = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t c = (w[i >> 2] >> (8 * (i & 3))) & 0x7fu;  // magnitude bits
        const uint32_t e = c >> 3, m = c & 7u;
        ok = ok && c != 0x7fu;
        // E4M3 magnitude: (1 + m/8) 2^(e-7), or m 2^-9 for e = 0
        const float a = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : static_cast<float>(m) * 0.001953125f;
        mx = fmaxf(mx, a);
      }
      const float s = eb ? __uint_as_float(eb << 23) : __uint_as_float(0x00400000u);
      return __all_sync(0xffffffffu, ok && mx * s < 65536.f);
    }
    const uint4* src = reinterpret_cast<const uint4*>(kv + row * kDqk);
    bool ok = true;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint4 v = __ldg(src + lane + 32 * k);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        ok = ok && (w[i] & 0x7fffu) < 0x4780u && ((w[i] >> 16) & 0x7fffu) < 0x4780u;
    }
    return __all_sync(0xffffffffu, ok);
  };
  for (int b = blockIdx.x; b < B; b += gridDim.x) {
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    const int L = lens[b];
    const int* row = bt + static_cast<long long>(b) * bt_stride;
    if (L < 0) {
      if (threadIdx.x == 0) atomicCAS(status, 0, static_cast<int>(kStBadTable));
    } else if (topk_idx == nullptr) {
      if (static_cast<long long>(L) > bt_stride * kPage) {
        if (threadIdx.x == 0) atomicCAS(status, 0, static_cast<int>(kStBadTable));
      } else {
        const int np = (L + kPage - 1) / kPage;
        for (int j = threadIdx.x; j < np; j += blockDim.x) {
          const int pg = row[j];
          if (pg < 0 || pg >= num_pages) {
            atomicCAS(status, 0, static_cast<int>(kStBadTable));
            s_bad = 1;
          }
        }
        __syncthreads();
        if (check_range && !s_bad) {
          for (int j = warp; j < L; j += nwarps) {
            const long long r = static_cast<long long>(row[j / kPage]) * kPage + j % kPage;
            if (!row_in_range(r)) {
              if (lane == 0) atomicCAS(status, 0, static_cast<int>(kStValueRange));
              break;
            }
          }
        }
      }
    } else {
      const int* ix = topk_idx + static_cast<long long>(b) * s_q * topk;
      for (int k = threadIdx.x; k < s_q * topk; k += blockDim.x) {
        const int v = ix[k];
        if (v < -1 || v >= L) {
          atomicCAS(status, 0, static_cast<int>(kStBadIndex));
          s_bad = 1;
        } else if (v >= 0) {
          const long long pi = v / kPage;
          if (pi >= bt_stride || row[pi] < 0 || row[pi] >= num_pages) {
            atomicCAS(status, 0, static_cast<int>(kStBadTable));
            s_bad = 1;
          }
        }
      }
      __syncthreads();
      if (check_range && !s_bad) {
        for (int k = warp; k < s_q * topk; k += nwarps) {
          const int v = ix[k];
          if (v < 0) continue;
          const long long r = static_cast<long long>(row[v / kPage]) * kPage + v % kPage;
          if (!row_in_range(r)) {
            if (lane == 0) atomicCAS(status, 0, static_cast<int>(kStValueRange));
            break;
          }
        }
      }
    }
    __syncthreads();  // s_bad is reset for the next request
  }
}

// ------------------------------------------------------------------ failure-path diagnostic
// One CTA waits, with the decode kernels' bounded wait, on a barrier that
// nothing completes; the wait records kStTimeout in *status and gives up.
__global__ void mla_wait_timeout_kernel(int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  Ctl ctl;
  ctl.abort = &abort_flag;
  ctl.n_remote = 0;
  ctl.status = status;
  if (threadIdx.x == 0) (void)wait_bar<false>(smem_u32(&bar), 0u, ctl);
  __syncthreads();
}

}  // namespace mla

