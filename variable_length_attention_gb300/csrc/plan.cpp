// plan.cpp -- host tile planners for the persistent kernels.
//
// Scheduling is decided on the CPU from the host copy of the offsets, so no
// device synchronisation is needed before a launch ("TLX Block Attention",
// section 5, scalar scheduling arithmetic on the CPU when CPU offsets exist).
//
// Forward: query work is split into units of 256 rows (two 128-row tiles that
// share every K/V load).  A unit's cost is the number of 128-key blocks it
// visits, which grows with the K/V length of its sequence.  Units are sorted by
// cost, largest first, and dealt to the CTAs in snake order -- left to right on
// even passes, right to left on odd ones -- so every CTA receives a mix of long
// and short work (aixai.ru summary, "Tile balancing and Cluster Launch Control").
//
// Backward: a unit is one valid 128-key block of one (sequence, key/value
// head); with grouped-query attention it visits the query tiles of every query
// head of its group, so the heads enumerated here are the key/value heads.  The
// pages describe the backward tiles as near-equal in cost with a varying count,
// so only valid blocks are listed and they are dealt round-robin, in an order
// where neighbouring tiles reuse the same data in L2 (same source, same
// section).  That holds for broadcast-Q, where every unit loops over the same
// shared query rows.  In self-attention a unit loops over the query tiles of
// its own sequence, so its cost grows with the sequence length; this planner
// therefore sorts units by cost (stably: equal costs keep the enumeration order
// sequence, head, block) and deals them in the same snake order as the
// forward.  With equal costs that is the pages' enumeration, dealt back and
// forth instead of strictly round-robin.
//
// Block-diagonal: BLOCK_PER_BATCH is the prefix sum of 64-token block counts;
// programs receive balanced contiguous ranges from closed-form divmod
// ("TLX Block Attention", section 5).  A tile here is a pair of consecutive
// global blocks for one head, because the tensor-core MMA used for it has 128
// rows (two 64-token blocks).
#include <algorithm>
#include <cstdint>
#include <vector>

#include "../../include/jfa.h"
#include "plan.h"

namespace jfa {

static inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

int check_offsets(const int32_t* offsets, int batch, int max_len) {
  if (offsets == nullptr || batch < 0) return JFA_ERR_INVALID_ARG;
  if (offsets[0] != 0) return JFA_ERR_BAD_OFFSETS;
  for (int b = 0; b < batch; ++b) {
    const int64_t L = static_cast<int64_t>(offsets[b + 1]) - offsets[b];
    if (L < 0) return JFA_ERR_BAD_OFFSETS;
    if (max_len >= 0 && L > max_len) return JFA_ERR_BAD_OFFSETS;
  }
  return JFA_OK;
}

// Both list planners share one dealing step.  Units arrive in enumeration
// order with a small integer cost.  A counting sort on the cost (largest first)
// gives the same order as a stable sort, in linear time: units of equal cost
// keep their enumeration order.  Sorted index t is dealt in pass p = t / P to
// slot r = t % P, CTA r on even passes and P-1-r on odd ones, so CTA c holds
// one unit per pass and the unit of pass p sits at position p of its list.
template <class Enumerate>
static int deal_sorted(Enumerate&& each, int64_t n, int n_cta, std::vector<int32_t>* units,
                       std::vector<int32_t>* cta_start) {
  if (units == nullptr && cta_start == nullptr) return static_cast<int>(n);
  const int64_t P = n_cta, full = n / P, rem = n % P;
  std::vector<int32_t> start(P + 1, 0);
  for (int64_t c = 0; c < P; ++c) {
    // the last, partial pass reaches CTAs 0..rem-1 (even pass) or P-rem..P-1 (odd pass)
    const bool extra = (full % 2 == 0) ? c < rem : c >= P - rem;
    start[c + 1] = static_cast<int32_t>(start[c] + full + (extra ? 1 : 0));
  }
  if (units) {
    int32_t max_cost = 0;
    each([&](int32_t, int32_t, int32_t, int32_t cost) { max_cost = std::max(max_cost, cost); });
    // bucket k holds cost max_cost - k; its cursor is the (pass, slot) of the
    // sorted index its next unit takes, advanced without a division per unit
    const size_t nb = static_cast<size_t>(max_cost) + 1;
    std::vector<int64_t> first(nb + 1, 0), pass(nb), slot(nb);
    each([&](int32_t, int32_t, int32_t, int32_t cost) { ++first[max_cost - cost + 1]; });
    for (size_t k = 1; k <= nb; ++k) first[k] += first[k - 1];
    for (size_t k = 0; k < nb; ++k) {
      pass[k] = first[k] / P;
      slot[k] = first[k] % P;
    }
    units->resize(4 * n);  // every entry is written below
    int32_t* out = units->data();
    each([&](int32_t b, int32_t h, int32_t m, int32_t cost) {
      const size_t k = static_cast<size_t>(max_cost - cost);
      const int64_t p = pass[k], r = slot[k];
      if (++slot[k] == P) {
        slot[k] = 0;
        ++pass[k];
      }
      const int64_t c = (p % 2 == 0) ? r : P - 1 - r;
      int32_t* e = out + 4 * (start[c] + p);
      e[0] = b;
      e[1] = h;
      e[2] = m;
      e[3] = cost;
    });
  }
  if (cta_start) *cta_start = std::move(start);
  return static_cast<int>(n);
}

// Visible keys of query row i: [i - left, i + right] inside the sequence, a
// negative bound leaving its side open (causal: left < 0, right = 0).
// K/V blocks the 256-row forward unit m visits: from the first block its first
// row sees to the last block its last row sees.
static int64_t fwd_unit_blocks(int64_t m, int64_t rows, int64_t L, int left, int right) {
  const int64_t r0 = kFwdRows * m, last = std::min<int64_t>(kFwdRows * (m + 1), rows) - 1;
  const int64_t lo = left < 0 ? 0 : std::max<int64_t>(0, r0 - left);
  const int64_t hi = right < 0 ? L : std::min<int64_t>(L, last + right + 1);
  return cdiv(hi, kKvBlock) - lo / kKvBlock;
}

// 128-row query tiles that the keys of 128-key block n meet.
static int64_t bwd_unit_tiles(int64_t n, int64_t rows, int64_t L, int left, int right) {
  const int64_t k_last = std::min<int64_t>(kKvBlock * (n + 1), L) - 1;
  const int64_t lo = right < 0 ? 0 : std::max<int64_t>(0, kKvBlock * n - right);
  const int64_t hi = left < 0 ? rows : std::min<int64_t>(rows, k_last + left + 1);
  return cdiv(hi, kKvBlock) - lo / kKvBlock;
}

int plan_fwd(const int32_t* offsets, int batch, int H, int nq, int causal, int n_cta, std::vector<int32_t>* units,
             std::vector<int32_t>* cta_start) {
  return plan_fwd_window(offsets, batch, H, nq, -1, causal ? 0 : -1, n_cta, units, cta_start);
}

int plan_fwd_window(const int32_t* offsets, int batch, int H, int nq, int left, int right, int n_cta,
                    std::vector<int32_t>* units, std::vector<int32_t>* cta_start) {
  // enumeration order: sequence, head, 256-row unit; cost = K/V blocks visited
  auto each = [&](auto&& fn) {
    for (int b = 0; b < batch; ++b) {
      const int64_t L = static_cast<int64_t>(offsets[b + 1]) - offsets[b];
      if (L == 0) continue;
      const int64_t rows = nq > 0 ? nq : L;
      const int64_t nm = cdiv(rows, kFwdRows);
      for (int h = 0; h < H; ++h)
        for (int64_t m = 0; m < nm; ++m)
          fn(b, h, static_cast<int32_t>(m), static_cast<int32_t>(fwd_unit_blocks(m, rows, L, left, right)));
    }
  };
  int64_t n = 0;
  for (int b = 0; b < batch; ++b) {
    const int64_t L = static_cast<int64_t>(offsets[b + 1]) - offsets[b];
    if (L > 0) n += static_cast<int64_t>(H) * cdiv(nq > 0 ? nq : L, kFwdRows);
  }
  return deal_sorted(each, n, n_cta, units, cta_start);
}

int plan_fwd_topk(const int32_t* offsets, int batch, int H, int nq, int topk, int n_cta, std::vector<int32_t>* units,
                  std::vector<int32_t>* cta_start) {
  // the forward's units and order; a unit visits its min(topk, blocks) chosen blocks
  auto each = [&](auto&& fn) {
    for (int b = 0; b < batch; ++b) {
      const int64_t L = static_cast<int64_t>(offsets[b + 1]) - offsets[b];
      if (L == 0) continue;
      const int64_t nm = cdiv(nq > 0 ? nq : L, kFwdRows);
      const int32_t cost = static_cast<int32_t>(std::min<int64_t>(topk, cdiv(L, kKvBlock)));
      for (int h = 0; h < H; ++h)
        for (int64_t m = 0; m < nm; ++m) fn(b, h, static_cast<int32_t>(m), cost);
    }
  };
  int64_t n = 0;
  for (int b = 0; b < batch; ++b) {
    const int64_t L = static_cast<int64_t>(offsets[b + 1]) - offsets[b];
    if (L > 0) n += static_cast<int64_t>(H) * cdiv(nq > 0 ? nq : L, kFwdRows);
  }
  return deal_sorted(each, n, n_cta, units, cta_start);
}

int plan_bwd(const int32_t* offsets, int batch, int H, int nq, int causal, int n_cta, std::vector<int32_t>* units,
             std::vector<int32_t>* cta_start) {
  return plan_bwd_window(offsets, batch, H, nq, -1, causal ? 0 : -1, n_cta, units, cta_start);
}

int plan_bwd_window(const int32_t* offsets, int batch, int H, int nq, int left, int right, int n_cta,
                    std::vector<int32_t>* units, std::vector<int32_t>* cta_start) {
  // enumeration order: sequence, head (key/value head), 128-key block; cost =
  // query tiles visited per query head.
  // Equal costs (broadcast-Q) keep this order; unequal ones (self-attention,
  // where a unit loops over its sequence's query tiles) come largest first so
  // the snake deal balances them.
  auto each = [&](auto&& fn) {
    for (int b = 0; b < batch; ++b) {
      const int64_t L = static_cast<int64_t>(offsets[b + 1]) - offsets[b];
      const int64_t rows = nq > 0 ? nq : L;
      const int64_t nblk = cdiv(L, kKvBlock);
      for (int h = 0; h < H; ++h)
        for (int64_t blk = 0; blk < nblk; ++blk)
          fn(b, h, static_cast<int32_t>(blk), static_cast<int32_t>(bwd_unit_tiles(blk, rows, L, left, right)));
    }
  };
  int64_t n = 0;
  for (int b = 0; b < batch; ++b)
    n += static_cast<int64_t>(H) * cdiv(static_cast<int64_t>(offsets[b + 1]) - offsets[b], kKvBlock);
  return deal_sorted(each, n, n_cta, units, cta_start);
}

int plan_block(const int32_t* offsets, int batch, int H, int n_sm, std::vector<int32_t>* bpb,
               std::vector<int32_t>* prog_start) {
  std::vector<int32_t> pre(batch + 1, 0);
  for (int b = 0; b < batch; ++b)
    pre[b + 1] = static_cast<int32_t>(pre[b] + cdiv(static_cast<int64_t>(offsets[b + 1]) - offsets[b], kBlk));
  const int64_t tiles = cdiv(pre[batch], 2) * H;
  const int64_t P = std::min<int64_t>(n_sm, tiles);
  if (prog_start) {
    prog_start->assign(P + 1, 0);
    if (P > 0) {
      const int64_t q = tiles / P, r = tiles % P;
      for (int64_t p = 0; p <= P; ++p) (*prog_start)[p] = static_cast<int32_t>(p * q + std::min(p, r));
    }
  }
  if (bpb) *bpb = pre;
  return static_cast<int>(P);
}

void units_for_device(std::vector<int32_t>* units, const int32_t* offsets) {
  for (size_t e = 0; e + 3 < units->size(); e += 4) {
    const int32_t b = (*units)[e];
    (*units)[e + 3] = offsets[b + 1] - offsets[b];
  }
}

}  // namespace jfa

// ------------------------------------------------------------- exported test hooks
extern "C" int jfa_plan_fwd(const int32_t* offsets_host, int batch, int num_heads, int nq_broadcast, int causal,
                            int n_cta, int32_t* units, int32_t* cta_start) {
  if (num_heads <= 0 || n_cta <= 0 || nq_broadcast < 0) return -JFA_ERR_INVALID_ARG;
  const int st = jfa::check_offsets(offsets_host, batch, -1);
  if (st != JFA_OK) return -st;
  std::vector<int32_t> u, s;
  const int n = jfa::plan_fwd(offsets_host, batch, num_heads, nq_broadcast, causal, n_cta, units ? &u : nullptr,
                              cta_start ? &s : nullptr);
  if (units) std::copy(u.begin(), u.end(), units);
  if (cta_start) std::copy(s.begin(), s.end(), cta_start);
  return n;
}

extern "C" int jfa_plan_bwd(const int32_t* offsets_host, int batch, int num_heads, int nq_broadcast, int causal,
                            int n_cta, int32_t* units, int32_t* cta_start) {
  if (num_heads <= 0 || n_cta <= 0 || nq_broadcast < 0) return -JFA_ERR_INVALID_ARG;
  const int st = jfa::check_offsets(offsets_host, batch, -1);
  if (st != JFA_OK) return -st;
  std::vector<int32_t> u, s;
  const int n = jfa::plan_bwd(offsets_host, batch, num_heads, nq_broadcast, causal, n_cta, units ? &u : nullptr,
                              cta_start ? &s : nullptr);
  if (units) std::copy(u.begin(), u.end(), units);
  if (cta_start) std::copy(s.begin(), s.end(), cta_start);
  return n;
}

extern "C" int jfa_plan_window(int which, const int32_t* offsets_host, int batch, int num_heads, int window_left,
                               int window_right, int n_cta, int32_t* units, int32_t* cta_start) {
  if (num_heads <= 0 || n_cta <= 0 || window_left < -1 || window_right < -1 || which < 0 || which > 1)
    return -JFA_ERR_INVALID_ARG;
  const int st = jfa::check_offsets(offsets_host, batch, -1);
  if (st != JFA_OK) return -st;
  std::vector<int32_t> u, s;
  int n;
  if (which == 0)
    n = jfa::plan_fwd_window(offsets_host, batch, num_heads, 0, window_left, window_right, n_cta,
                             units ? &u : nullptr, cta_start ? &s : nullptr);
  else
    n = jfa::plan_bwd_window(offsets_host, batch, num_heads, 0, window_left, window_right, n_cta,
                             units ? &u : nullptr, cta_start ? &s : nullptr);
  if (units) std::copy(u.begin(), u.end(), units);
  if (cta_start) std::copy(s.begin(), s.end(), cta_start);
  return n;
}

extern "C" int block_plan(const int32_t* offsets_host, int batch, int num_heads, int n_sm,
                          int32_t* block_per_batch, int32_t* prog_start) {
  if (num_heads <= 0 || n_sm <= 0) return -JFA_ERR_INVALID_ARG;
  const int st = jfa::check_offsets(offsets_host, batch, -1);
  if (st != JFA_OK) return -st;
  std::vector<int32_t> b, p;
  const int P = jfa::plan_block(offsets_host, batch, num_heads, n_sm, &b, &p);
  if (block_per_batch) std::copy(b.begin(), b.end(), block_per_batch);
  if (prog_start) std::copy(p.begin(), p.end(), prog_start);
  return P;
}
