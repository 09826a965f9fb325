// plan.cuh — split-KV partition of a decode step (shared by the device plan
// kernel and the host mirror).
//
// Work unit: one tile of one request: 64 cached rows, or 128 on the
// two-token dense path (whose tiles are two pages; see plan_tile_rows).
// Request b has n_b = ceil(len_b / rows) tiles (ceil(topk / 64) for top-k
// lists) and costs n_b + C0 when n_b > 0, C0 standing for the per-split fixed
// work (loading the query block and writing the output block).  Requests
// are laid end to end on a cost line; unit u owns the cost interval
// [u*W, (u+1)*W), W = max(ceil(total / U), MIN_W).  A cut that falls inside
// a request's fixed-cost prefix snaps to the request start; a cut inside its
// tiles splits it.  This is the persistent-grid form of choosing the split
// count so that no partial wave is left ("The Premise That Wasn't",
// Wave-Aware NSPLIT): every unit gets the same load, so there is no tail.
#pragma once
#include <cstdint>

namespace mla {

constexpr int kPlanC0 = 2;       // fixed cost of a split, in tiles
constexpr int kPlanMinTiles = 4; // a unit takes at least this many tiles

struct ReqInfo {   // per request, int4 in the workspace
  int n_tiles;     // tiles (64 or 128 rows, see plan_tile_rows)
  int n_splits;    // units touching it (0 = nothing to attend to)
  int first_slot;  // partial-result slot of split 0 (only if n_splits > 1)
  int cost_prefix; // exclusive prefix of costs
};

struct UnitInfo {  // per unit, 5 ints in the workspace
  int begin_req, begin_tile, end_req, end_tile, first_split;
};

// Rows per tile: the two-token (s_q = 2) dense kernel walks two pages at a
// time; every other path one page (or 64 top-k entries).
__host__ __device__ inline int plan_tile_rows(int s_q, int topk) {
  return (s_q == 2 && topk == 0) ? 128 : 64;
}

__host__ __device__ inline int plan_tiles(int len, int topk, int tile_rows) {
  if (topk > 0) return (topk + 63) / 64;
  return len > 0 ? (len + tile_rows - 1) / tile_rows : 0;
}

__host__ __device__ inline int plan_cost(int n_tiles) { return n_tiles > 0 ? n_tiles + kPlanC0 : 0; }

__host__ __device__ inline int plan_width(int total_cost, int num_units) {
  int w = (total_cost + num_units - 1) / num_units;
  int lo = kPlanC0 + kPlanMinTiles;
  return w > lo ? w : lo;
}

__host__ __device__ inline int ceil_div_pos(int a, int b) { return a <= 0 ? 0 : (a + b - 1) / b; }

// Number of units that touch request b (0 if it has no tiles).
__host__ __device__ inline int plan_n_splits(int prefix, int n_tiles, int W, int U) {
  if (n_tiles <= 0) return 0;
  // cuts k*W (1 <= k <= U-1) with prefix + C0 + 1 <= k*W <= prefix + C0 + n_tiles - 1
  int lo = ceil_div_pos(prefix + kPlanC0 + 1, W);
  if (lo < 1) lo = 1;
  int hi = (prefix + kPlanC0 + n_tiles - 1) / W;
  if (hi > U - 1) hi = U - 1;
  return 1 + (hi >= lo ? hi - lo + 1 : 0);
}

// (request, tile) at cost x: the last request whose prefix is <= x.
// `prefix(b)` is a callable giving the exclusive cost prefix of request b.
template <typename PrefixFn>
__host__ __device__ inline void plan_position(int x, int total, int B, PrefixFn prefix,
                                              int& req, int& tile) {
  if (x >= total) { req = B; tile = 0; return; }
  int lo = 0, hi = B - 1;  // find last b with prefix(b) <= x
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (prefix(mid) <= x) lo = mid; else hi = mid - 1;
  }
  req = lo;
  int t = x - prefix(lo) - kPlanC0;
  tile = t > 0 ? t : 0;
}

template <typename PrefixFn>
__host__ __device__ inline UnitInfo plan_unit(int u, int W, int total, int B, PrefixFn prefix) {
  UnitInfo ui;
  long long xb = static_cast<long long>(u) * W;
  long long xe = xb + W;
  int b0 = xb < total ? static_cast<int>(xb) : total;
  int e0 = xe < total ? static_cast<int>(xe) : total;
  plan_position(b0, total, B, prefix, ui.begin_req, ui.begin_tile);
  plan_position(e0, total, B, prefix, ui.end_req, ui.end_tile);
  ui.first_split = 0;
  if (ui.begin_req < B && ui.begin_tile > 0) {
    int k_first = ceil_div_pos(prefix(ui.begin_req) + kPlanC0 + 1, W);
    ui.first_split = u - k_first + 1;
  }
  return ui;
}

}  // namespace mla
