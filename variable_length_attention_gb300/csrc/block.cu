// block.cu -- fixed 64-token block-diagonal attention for sm_103a.
//
// What it computes ("TLX Block Attention", sections 1 and 2.1): every sequence
// is cut into blocks of 64 tokens (the last one may be shorter) and each block
// attends only within itself.  Because a query block meets exactly one key
// block, the score tile is complete after one GEMM: the row max and sum are
// final at once, so there is no running-max correction, no stored log-sum-exp
// and every accumulator starts fresh (use_acc = false).  The backward (section 4)
// recomputes P from Q and K, forms Di = rowsum(P o dP) inline, and every block
// owns its own dQ, dK and dV rows, so nothing is reduced across CTAs.
//
// Rotary variants (a template parameter): each tile's Q and K are rotated in
// shared memory as soon as TMA has landed them, by warps of their own (four
// added to the forward's, two otherwise idle ones in the backward), from a
// packed fp16 cos/sin table the
// entry point builds per call (rope.cu), and the score GEMM waits for them.  The
// backward's dQ and dK go back through the transposed rotation in its epilogue,
// each thread on its own fp32 row as it comes out of TMEM, before rounding.
//
// Tiles: the tensor-core MMA used here has 128 rows, so a tile stacks two
// consecutive global blocks (2p, 2p+1) of one head: rows 0-63 are block 2p,
// rows 64-127 block 2p+1, and the off-diagonal quadrants of the 128 x 128 score
// tile are masked.  That doubles the tensor work, which is free here: the kernel
// moves ~33 FLOP per byte, far below the ridge, so it is bound by HBM
// ("TLX Block Attention", section 3.3).  Persistent programs take balanced
// contiguous ranges of (pair, head) tiles from the host plan, or, under
// Cluster Launch Control, chunks of consecutive tiles: one CTA per chunk is
// launched and a CTA that finishes a chunk cancels the launch of a CTA not yet
// running and takes its chunk, so imbalance that shows only at run time is
// absorbed ("TLX Block Attention", section 5; aixai.ru summary, "Tile balancing
// and Cluster Launch Control").  The sequence of a global block is found by a
// branchless binary search over the per-batch block prefix sums (section 5),
// which each role runs only when its tiles leave the sequence it found last.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "block.h"
#include "host.h"
#include "profile.h"
#include "ptx.cuh"

namespace jfa {
namespace blk {

constexpr int kBlk = 64;
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
  const int32_t* offsets;
  const int32_t* bpb;         // [batch+1] prefix sums of blocks per sequence
  const int32_t* prog_start;  // [P+1] (static ranges)
  int* err;
  __nv_bfloat16 *o, *dq, *dk, *dv;
  int batch, H, n_blocks;
  float scale, scale_log2;
  int use_clc;                // 1: one CTA per chunk of `chunk` tiles, Cluster Launch Control
  int chunk, n_tiles, n_chunks;
  const uint32_t* rope_tab;   // rotary variant: packed table, [positions, D/2] words (rope.h:
                              // word 2m: cos of pairs 2m, 2m+1 as half2; word 2m+1: their sines)
};

// Tiles [*tb, *te) of schedule entry `ch`: chunk ch under Cluster Launch
// Control, else the CTA's own static range.
__device__ __forceinline__ void chunk_range(const Params& p, int ch, int* tb, int* te) {
  if (p.use_clc) {
    *tb = ch * p.chunk;
    *te = min(*tb + p.chunk, p.n_tiles);
  } else {
    *tb = p.prog_start[blockIdx.x];
    *te = p.prog_start[blockIdx.x + 1];
  }
}

// The tiles a CTA works on, in order, as every role sees them: the loader
// publishes schedule entries (chunks) through the 4-slot ring; each consumer
// walks the tiles of the entries it pops.
struct TileCursor {
  int t = 0, te = 0;
  uint32_t sit = 0;
};
// Next tile id; -1 at the end, -2 if the CTA aborts.
template <class Bars>
__device__ __forceinline__ int next_tile(TileCursor& c, Bars* bars, const Params& p, const Abort& ab, bool per_warp) {
  while (c.t >= c.te) {
    const int ch = sched_pop(bars, c.sit++, ab, per_warp);
    if (ch < 0) return ch;
    chunk_range(p, ch, &c.t, &c.te);
  }
  return c.t++;
}

// The loader's side of the schedule: publishes entry `cur` in ring slot `sit`,
// and under Cluster Launch Control asks for a CTA not yet launched.  Returns
// false if the CTA aborts.
template <class Bars>
__device__ __forceinline__ bool publish(Bars* bars, uint32_t sit, int cur, const Params& p, const Abort& ab) {
  const int slot = sit & 3;
  if (!mbar_wait(&bars->sched_empty[slot], ((sit >> 2) & 1) ^ 1, ab)) return false;
  bars->sched_unit[slot] = cur;
  mbar_arrive(&bars->sched_full[slot]);
  if (cur >= 0 && p.use_clc) {
    mbar_expect_tx(&bars->clc_bar, 16);
    clc_try_cancel(&bars->clc_resp, &bars->clc_bar);
  }
  return true;
}
// The entry after `sit`'s: the cancelled CTA's chunk, or -1 (also -1 under the
// static ranges, which have one entry); -2 if the CTA aborts.
template <class Bars>
__device__ __forceinline__ int next_entry(Bars* bars, uint32_t sit, const Params& p, const Abort& ab) {
  if (!p.use_clc) return -1;
  if (!mbar_wait(&bars->clc_bar, sit & 1, ab)) return -2;
  const int nxt = clc_cancelled_x(&bars->clc_resp);
  return nxt >= p.n_chunks ? -1 : nxt;
}

// One 64-token block: first token row and length (0 if the block does not exist).
struct Blk {
  int row0, len;
  int pos0;  // position of the block's first row inside its sequence
};

// Global block g -> its rows.  Each role walks the tiles in ascending block
// order, the heads of a pair one after another and most pairs inside the
// sequence of the previous one, so the sequence found last is kept and the
// search (a chain of dependent loads) runs only when g leaves it.
struct Locator {
  int g_lo = 0, g_hi = 0;  // blocks [g_lo, g_hi) are those of the kept sequence
  int s = 0, L = 0;        // its first row and length
  __device__ __forceinline__ Blk operator()(const Params& p, int g) {
    Blk r{0, 0, 0};
    if (g >= p.n_blocks) return r;
    if (g < g_lo || g >= g_hi) {
      // largest b in [0, batch) with bpb[b] <= g (branchless halving search)
      int lo = 0, n = p.batch;
      while (n > 1) {
        const int half = n >> 1;
        lo = (__ldg(p.bpb + lo + half) <= g) ? lo + half : lo;
        n -= half;
      }
      g_lo = __ldg(p.bpb + lo);
      g_hi = __ldg(p.bpb + lo + 1);
      s = __ldg(p.offsets + lo);
      L = __ldg(p.offsets + lo + 1) - s;
    }
    const int j = g - g_lo;
    r.row0 = s + kBlk * j;
    r.len = min(kBlk, L - kBlk * j);
    r.pos0 = kBlk * j;
    return r;
  }
};

// Byte offset of column c of row `row` in a tile of 128-byte-swizzled 64-column boxes.
template <int D>
__device__ __forceinline__ uint32_t rot_off(int row, int c) {
  return (c / 64) * 16384 + row * 128 + ((((c % 64) / 8) ^ (row & 7)) << 4);
}
// Two column pairs of a row: u holds elements (i, i+1) of the first half, v
// their partners (i + D/2, i + 1 + D/2), c and s the pairs' cosines and sines;
// the rotation turns (u, v) into (u c - v s, v c + u s), its transpose into
// (u c + v s, v c - u s), in paired fp32 arithmetic.
template <bool TRANSPOSED>
__device__ __forceinline__ void rot2(uint64_t u, uint64_t v, uint64_t c, uint64_t s, uint64_t& uo, uint64_t& vo) {
  const uint64_t ns = fmul2(s, f32x2(-1.0f, -1.0f));
  uo = ffma2(v, TRANSPOSED ? s : ns, fmul2(u, c));
  vo = ffma2(u, TRANSPOSED ? ns : s, fmul2(v, c));
}
__device__ __forceinline__ uint64_t h2_to_f32x2(uint32_t w) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
  return f32x2(f.x, f.y);
}
__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t w) {
  return f32x2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(uint64_t r) {
  float lo, hi;
  f32x2_split(r, lo, hi);
  return pack_bf16(lo, hi);
}
// Rotates Q and K rows [r0, r0 + NROWS) of one 64-row half of a tile pair in place, each tile
// stored as D/64 128-byte-swizzled 64-column boxes: for i < D/2 the pair
// (x_i, x_{i+D/2}) becomes (x_i c_i - x_{i+D/2} s_i, x_{i+D/2} c_i + x_i s_i), c and
// s from the packed table row of the row's position.  One warp: each lane takes
// a 16-byte chunk of the first half of a row (columns 8j..8j+7) and its partner
// chunk of the second half, 4 rows per step at D = 128 (8 at D = 64).  Steps go
// in batches of B: the batch's shared-memory loads are all issued before its
// stores, and the next batch's table rows load while this one is rotated, so
// neither the shared-memory nor the table latency is paid per row.  Rows past
// the block's end are left alone (their scores are masked).
// `ready` is called once the first batch's table rows are on their way (it waits
// for the tile to land, so the table latency overlaps that wait); false aborts.
struct NoWait {
  __device__ bool operator()() const { return true; }
};
template <int D, int NROWS, int B, class Ready = NoWait>
__device__ __forceinline__ bool rope_rows(const uint32_t* __restrict__ tab, uint8_t* q_tile, uint8_t* k_tile,
                                          int half, int r0, const Blk& blk, int lane, Ready ready = Ready()) {
  constexpr int CPR = D / 16;    // chunks in half a row
  constexpr int RPS = 32 / CPR;  // rows per step; B steps per batch
  constexpr int NB = NROWS / RPS / B;
  constexpr int NT = 2;          // tensors: q and k
  const int j = lane % CPR, sub = lane / CPR;
  const int c1 = 8 * j, c2 = 8 * j + D / 2;
  const uint32_t base[2] = {smem_u32(q_tile), smem_u32(k_tile)};
  uint4 t[2][B][2];  // table words of the chunk's 8 pairs: [buffer][step][pairs 0-3 | 4-7]
  auto load_tab = [&](int bi, int buf) {
#pragma unroll
    for (int st = 0; st < B; ++st) {
      const int rr = r0 + (bi * B + st) * RPS + sub;
      if (rr < blk.len) {
        const uint4* e = reinterpret_cast<const uint4*>(tab + static_cast<size_t>(blk.pos0 + rr) * (D / 2) + c1);
        t[buf][st][0] = __ldg(e);
        t[buf][st][1] = __ldg(e + 1);
      }
    }
  };
  load_tab(0, 0);
  if (!ready()) return false;
#pragma unroll
  for (int bi = 0; bi < NB; ++bi) {
    const int buf = bi & 1;
    if (bi + 1 < NB) load_tab(bi + 1, buf ^ 1);
    uint4 x[B][NT], y[B][NT];
#pragma unroll
    for (int st = 0; st < B; ++st) {
      const int rr = r0 + (bi * B + st) * RPS + sub;
      if (rr < blk.len) {
        const int row = 64 * half + rr;
#pragma unroll
        for (int tn = 0; tn < NT; ++tn) {
          const uint32_t a1 = base[tn] + rot_off<D>(row, c1), a2 = base[tn] + rot_off<D>(row, c2);
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(x[st][tn].x), "=r"(x[st][tn].y), "=r"(x[st][tn].z), "=r"(x[st][tn].w) : "r"(a1));
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(y[st][tn].x), "=r"(y[st][tn].y), "=r"(y[st][tn].z), "=r"(y[st][tn].w) : "r"(a2));
        }
      }
    }
#pragma unroll
    for (int st = 0; st < B; ++st) {
      const int rr = r0 + (bi * B + st) * RPS + sub;
      if (rr < blk.len) {
        const int row = 64 * half + rr;
        // word pairs (cos of pairs 2w, 2w+1; their sin)
        const uint4* tt = t[buf][st];
        const uint64_t cw[4] = {h2_to_f32x2(tt[0].x), h2_to_f32x2(tt[0].z), h2_to_f32x2(tt[1].x), h2_to_f32x2(tt[1].z)};
        const uint64_t sw[4] = {h2_to_f32x2(tt[0].y), h2_to_f32x2(tt[0].w), h2_to_f32x2(tt[1].y), h2_to_f32x2(tt[1].w)};
#pragma unroll
        for (int tn = 0; tn < NT; ++tn) {
          const uint32_t xi[4] = {x[st][tn].x, x[st][tn].y, x[st][tn].z, x[st][tn].w};
          const uint32_t yi[4] = {y[st][tn].x, y[st][tn].y, y[st][tn].z, y[st][tn].w};
          uint32_t xo[4], yo[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            uint64_t uo, vo;
            rot2<false>(bf16x2_to_f32x2(xi[w]), bf16x2_to_f32x2(yi[w]), cw[w], sw[w], uo, vo);
            xo[w] = f32x2_to_bf16x2(uo);
            yo[w] = f32x2_to_bf16x2(vo);
          }
          const uint32_t a1 = base[tn] + rot_off<D>(row, c1), a2 = base[tn] + rot_off<D>(row, c2);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a1), "r"(xo[0]), "r"(xo[1]), "r"(xo[2]),
                       "r"(xo[3]) : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a2), "r"(yo[0]), "r"(yo[1]), "r"(yo[2]),
                       "r"(yo[3]) : "memory");
        }
      }
    }
  }
  return true;
}

// The rotation role of the rotary variants: every tile's Q and K once their
// slot has landed, rows [r0, r0 + NROWS) of the tile's first (half 0) or second
// (half 1) block; the score GEMM waits for qk_rot.  The forward runs four such
// warps (32 rows each), the backward two (a whole block each).
template <int D, int NQK, int NROWS, int B, class Bars>
__device__ __forceinline__ void rope_role(const Params& p, Bars* bars, uint8_t* smem, int tile_bytes, int half, int r0,
                                          const Abort& ab) {
  const int lane = lane_id();
  TileCursor cur;
  Locator locate;
  for (int i = 0;; ++i) {
    const int t = next_tile(cur, bars, p, ab, true);
    if (t < 0) break;
    const int st = i % NQK;
    uint8_t* q_tile = smem + st * 2 * tile_bytes;
    if (!rope_rows<D, NROWS, B>(p.rope_tab, q_tile, q_tile + tile_bytes, half, r0, locate(p, 2 * (t / p.H) + half),
                                lane, [&] { return mbar_wait(&bars->qk_full[st], (i / NQK) & 1, ab); }))
      break;
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->qk_rot[st]);
  }
}

// Operands come in two rings: Q and K of a tile together (released as soon as
// its score GEMM has read them) and V on its own (released after the PV GEMM),
// so more bytes are in flight from HBM than with whole Q/K/V stages.
template <int D>
struct FwdCfg {
  static constexpr int TILE = 128 * D * 2;         // 128 rows x D, bf16
  static constexpr int CHUNK = 128 * 128;          // 64 columns x 128 rows
  // Q+K and V slots: at D = 128 two and three fill the 227 KB; at D = 64 four
  // and four (192 KB) measured fastest of the splits tried (two and six, three
  // and four, three and three, four and two)
  static constexpr int NQK = D == 128 ? 2 : 4;
  static constexpr int NV = D == 128 ? 3 : 4;
  static constexpr int OFF_V = NQK * 2 * TILE;
  static constexpr int OFF_BAR = OFF_V + NV * TILE;
  static constexpr int SMEM = OFF_BAR + 512 + 1024;  // + alignment slack
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct FwdBars {
  int4 clc_resp;  // Cluster Launch Control response (16-byte aligned)
  uint64_t qk_full[4], qk_empty[4], v_full[4], v_empty[4];
  uint64_t qk_rot[4];  // rotary variant: Q and K of the slot are rotated
  uint64_t s_full[2], p_full[2], o_full[2], t_free[2];
  uint64_t drain;
  uint64_t sched_full[4], sched_empty[4], clc_bar;  // schedule ring (chunks), see publish()
  int sched_unit[4];
  uint32_t tmem_base;
  int abort_flag;
};
// the MMA thread and the 8 softmax warps (and the rotary variant's 4 rotation warps)
constexpr int kFwdSchedConsumers = 9;

// Loads rows [row0, row0+64) of every 64-column chunk of head h into rows
// [64*half, 64*half+64) of a 128-row swizzled tile.
template <int D>
__device__ __forceinline__ void load_half(const CUtensorMap* tm, uint64_t* bar, uint8_t* tile, int half, int h, int row0) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) tma_load_2d(tm, bar, tile + c * 16384 + half * 8192, h * D + c * 64, row0);
}

template <int D, bool ROPE>
__global__ void __launch_bounds__(ROPE ? 512 : 384, 1)
    block_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const Params p) {
  using C = FwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  FwdBars* bars = reinterpret_cast<FwdBars*>(smem + C::OFF_BAR);
  static_assert(C::NQK <= 4 && C::NV <= 4, "barrier arrays of the slot rings");
  static_assert(sizeof(FwdBars) <= 512, "barrier block");
  const int warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bars->sched_full[s], 1);
      mbar_init(&bars->sched_empty[s], kFwdSchedConsumers + (ROPE ? 4 : 0));
    }
    mbar_init(&bars->clc_bar, 1);
    for (int s = 0; s < C::NQK; ++s) {
      mbar_init(&bars->qk_full[s], 1);
      mbar_init(&bars->qk_empty[s], 1);
      mbar_init(&bars->qk_rot[s], 4);  // the 4 rotation warps
    }
    for (int s = 0; s < C::NV; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->p_full[b], 4);
      mbar_init(&bars->o_full[b], 1);
      mbar_init(&bars->t_free[b], 4);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const Abort ab{&bars->abort_flag, p.err};

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- loader and scheduler
    // In the order the tensor core consumes them: QK(0), then QK(i+1), V(i),
    // across chunk boundaries.  Consecutive tiles share their pair of blocks
    // across the heads, so the block search runs once per pair, not per load.
    int cached_pair = -1;
    Blk ca{0, 0}, cb{0, 0};
    Locator locate;
    auto rows = [&](int t, Blk& a, Blk& b, int& h) {
      const int pair = t / p.H;
      h = t % p.H;
      if (pair != cached_pair) {
        cached_pair = pair;
        ca = locate(p, 2 * pair);
        cb = locate(p, 2 * pair + 1);
        if (cb.len == 0) cb = ca;  // nothing there: reload block a, masked later
      }
      a = ca;
      b = cb;
    };
    auto load_qk = [&](int i, int t) -> bool {
      const int st = i % C::NQK;
      if (!mbar_wait(&bars->qk_empty[st], ((i / C::NQK) & 1) ^ 1, ab)) return false;
      Blk a, b;
      int h;
      rows(t, a, b, h);
      uint8_t* base = smem + st * 2 * C::TILE;
      mbar_expect_tx(&bars->qk_full[st], 2 * C::TILE);
      load_half<D>(&tm_q, &bars->qk_full[st], base, 0, h, a.row0);
      load_half<D>(&tm_q, &bars->qk_full[st], base, 1, h, b.row0);
      load_half<D>(&tm_k, &bars->qk_full[st], base + C::TILE, 0, h, a.row0);
      load_half<D>(&tm_k, &bars->qk_full[st], base + C::TILE, 1, h, b.row0);
      return true;
    };
    auto load_v = [&](int i, int t) -> bool {
      const int st = i % C::NV;
      if (!mbar_wait(&bars->v_empty[st], ((i / C::NV) & 1) ^ 1, ab)) return false;
      Blk a, b;
      int h;
      rows(t, a, b, h);
      uint8_t* base = smem + C::OFF_V + st * C::TILE;
      mbar_expect_tx(&bars->v_full[st], C::TILE);
      load_half<D>(&tm_v, &bars->v_full[st], base, 0, h, a.row0);
      load_half<D>(&tm_v, &bars->v_full[st], base, 1, h, b.row0);
      return true;
    };
    int cur = p.use_clc ? static_cast<int>(blockIdx.x) : 0;
    int i = 0, prev_t = -1;  // tiles loaded so far; the tile whose V is still to load
    for (uint32_t sit = 0;; ++sit) {
      if (!publish(bars, sit, cur, p, ab) || cur < 0) break;
      int tb, te;
      chunk_range(p, cur, &tb, &te);
      bool ok = true;
      for (int t = tb; t < te && ok; ++t, ++i) {
        ok = load_qk(i, t) && (prev_t < 0 || load_v(i - 1, prev_t));
        prev_t = t;
      }
      if (!ok) break;
      cur = next_entry(bars, sit, p, ab);
      if (cur == -2) break;
      if (cur < 0 && prev_t >= 0) load_v(i - 1, prev_t);  // the last tile's V
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    const uint32_t id_s = idesc_bf16(128, 128, 0, 0), id_o = idesc_bf16(128, D, 0, 1);
    const uint32_t sb = smem_u32(smem);
    auto issue_s = [&](int i) {
      const int st = i % C::NQK, b = i & 1;
      const uint32_t q = sb + st * 2 * C::TILE, k = q + C::TILE;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
        mma_ss(tmem + 256 * b, sdesc_sw128(q + off, 16, 1024), sdesc_sw128(k + off, 16, 1024), id_s, kk > 0);
      }
      mma_commit(&bars->s_full[b]);
      mma_commit(&bars->qk_empty[st]);  // Q and K are read: the slot may refill
    };
    auto issue_pv = [&](int i) {
      const int st = i % C::NV, b = i & 1;
      const uint32_t v = sb + C::OFF_V + st * C::TILE;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ts(tmem + 256 * b + 128, tmem + 256 * b + 8 * kk, sdesc_sw128(v + kk * 2048, C::CHUNK, 1024), id_o,
               kk > 0);
      mma_commit(&bars->o_full[b]);
      mma_commit(&bars->v_empty[st]);
    };
    TileCursor cur;
    for (int i = 0;; ++i) {
      const int t = next_tile(cur, bars, p, ab, false);
      if (t == -2) break;
      if (t >= 0) {  // S of tile i, once its operands landed (and are rotated) and its TMEM buffer is free
        if (!mbar_wait(ROPE ? &bars->qk_rot[i % C::NQK] : &bars->qk_full[i % C::NQK], (i / C::NQK) & 1, ab)) break;
        if (!mbar_wait(&bars->t_free[i & 1], ((i >> 1) & 1) ^ 1, ab)) break;
        tc_fence_after();
        issue_s(i);
      }
      if (i > 0) {  // PV of tile i-1
        const int j = i - 1;
        if (!mbar_wait(&bars->p_full[j & 1], (j >> 1) & 1, ab)) break;
        if (!mbar_wait(&bars->v_full[j % C::NV], (j / C::NV) & 1, ab)) break;
        tc_fence_after();
        issue_pv(j);
      }
      if (t < 0) break;
    }
    mma_commit(&bars->drain);
    const uint64_t tw = global_timer_ns();
    while (!mbar_try_wait(&bars->drain, 0) && global_timer_ns() - tw < kWaitTimeoutNs) {
    }
  } else if (ROPE && warp >= 12) {
    // ---------------------------------------------------------------- rotation (rotary variant)
    // warps 12-15: rows 0-31 / 32-63 of the tile's first block, then its second
    rope_role<D, C::NQK, 32, 2>(p, bars, smem, C::TILE, (warp - 12) >> 1, 32 * (warp & 1), ab);
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- softmax + epilogue
    const int b = (warp - 4) >> 2;          // TMEM buffer / tile parity of this warpgroup
    const int r = threadIdx.x & 127;        // row of the tile == TMEM lane
    const int half = r >> 6;
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_addr + 256 * b;
    const uint32_t tO = tS + 128;
    const float sl2 = p.scale_log2;
    TileCursor cur;
    Locator locate;
    for (int i = 0;; ++i) {
      const int t = next_tile(cur, bars, p, ab, true);
      if (t == -2) goto done;
      if (t < 0) break;
      if ((i & 1) != b) continue;  // the other warpgroup's tile
      const int pair = t / p.H, h = t % p.H;
      const Blk blk = locate(p, 2 * pair + half);
      const int rr = r & 63;
      if (!mbar_wait(&bars->s_full[b], (i >> 1) & 1, ab)) goto done;
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld32(tS + 64 * half, sr);
      tmem_ld32(tS + 64 * half + 32, sr + 32);
      tmem_wait_ld();
      reg_fence<64>(sr);
      float s[64];
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        s[c] = c < blk.len ? __uint_as_float(sr[c]) * sl2 : -INFINITY;
        mx = fmaxf(mx, s[c]);
      }
      if (blk.len == 0) mx = 0.f;
      float l = 0.f;
      uint32_t pk[32], zero[32];
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float p0 = ex2(s[c] - mx), p1 = ex2(s[c + 1] - mx);
        l += p0 + p1;
        pk[c / 2] = pack_bf16(p0, p1);
        zero[c / 2] = 0u;
      }
      // P packed two per column: keys of this row's block, zeros elsewhere
      tmem_st32(tS + 32 * half, pk);
      tmem_st32(tS + 32 * (1 - half), zero);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[b]);
      if (!mbar_wait(&bars->o_full[b], (i >> 1) & 1, ab)) goto done;
      tc_fence_after();
      const bool valid = rr < blk.len;
      const float inv_l = l > 0.f ? 1.0f / l : 0.f;
      __nv_bfloat16* dst = p.o + (static_cast<size_t>(blk.row0 + rr) * p.H + h) * D;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t ov[32];
        tmem_ld32(tO + c, ov);
        tmem_wait_ld();
        reg_fence<32>(ov);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = pack_bf16(__uint_as_float(ov[2 * e]) * inv_l, __uint_as_float(ov[2 * e + 1]) * inv_l);
        if (valid) {
#pragma unroll
          for (int e = 0; e < 4; ++e) st_global_v4(dst + c + 8 * e, w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->t_free[b]);
    }
  }
done:
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ backward
// Operands by lifetime: Q and K (read until the last GEMM) in a 2-slot ring, so
// the next tile's pair loads during this tile; V and dO (last read by the dV
// GEMM) in one slot that refills from the middle of the tile; P and then dS
// share one buffer (dS is written once the dV GEMM has read P).
template <int D>
struct BwdCfg {
  // D = 64 runs a separate epilogue warpgroup (warps 8-11) on accumulators of
  // their own in TMEM, so one tile's stores overlap the next tile's GEMMs and
  // softmax; at D = 128 the accumulators share TMEM with S and dP (no room for
  // both) and the softmax warps run the epilogue themselves.
  static constexpr bool SPLIT = D == 64;
  static constexpr int THREADS = SPLIT ? 384 : 256;
  static constexpr int TILE = 128 * D * 2;
  static constexpr int CHUNK = 128 * 128;
  static constexpr int NQK = SPLIT ? 3 : 2;         // Q,K slots
  static constexpr int NVD = SPLIT ? 2 : 1;         // V,dO slots
  static constexpr int OFF_V = NQK * 2 * TILE;      // slot s: V at OFF_V + 2 s TILE, dO one TILE later
  static constexpr int OFF_PDS = OFF_V + NVD * 2 * TILE;  // P, then dS: [128 q][128 keys] bf16
  static constexpr int OFF_BAR = OFF_PDS + 32768;
  static constexpr int SMEM = OFF_BAR + 512 + 1024;
  // TMEM columns: S [0,128), dP [128,256), dV [256, 256+D); dK and dQ go into
  // the dP and S columns (D = 128) or after dV (D = 64)
  static constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256;
  static constexpr uint32_t COL_DK = SPLIT ? 256 + D : COL_DP, COL_DQ = SPLIT ? 256 + 2 * D : COL_S;
  static constexpr int SCHED_CONSUMERS = SPLIT ? 9 : 5;  // the MMA thread and the 4 (or 8) consumer warps
};

struct BwdBars {
  int4 clc_resp;  // Cluster Launch Control response (16-byte aligned)
  uint64_t qk_full[3], qk_empty[3], vdo_full[2], vdo_empty[2];
  uint64_t qk_rot[3];  // rotary variant: Q and K of the slot are rotated
  uint64_t s_full, dp_full, p_full, p_used, ds_full, acc_full, t_free;
  uint64_t stg_free;  // D = 128 epilogue: every staged box read out by TMA (the next P may go in)
  uint64_t box_full[2], box_free[2];  // the same buffer per 64-column box: rows written / read out
  uint64_t drain;
  uint64_t sched_full[4], sched_empty[4], clc_bar;  // schedule ring (chunks), see publish()
  int sched_unit[4];
  uint32_t tmem_base;
  int abort_flag;
};

// Row q of a [128][128] bf16 tile stored as two swizzled 64-column boxes:
// 16-byte piece j (columns 8j..8j+7) of box c.
__device__ __forceinline__ void st_row_piece(uint8_t* tile, int q, int c, int j, const uint32_t* w) {
  const uint32_t addr = smem_u32(tile + c * 16384 + q * 128 + ((j ^ (q & 7)) << 4));
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
               : "memory");
}

template <int D, bool ROPE>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    block_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                     const __grid_constant__ CUtensorMap tm_dv, const Params p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::OFF_BAR);
  static_assert(C::NQK <= 3 && C::NVD <= 2, "barrier arrays of the slot rings");
  static_assert(sizeof(BwdBars) <= 512, "barrier block");
  const int warp = warp_id(), lane = lane_id();
  constexpr uint32_t COL_S = C::COL_S, COL_DP = C::COL_DP, COL_DV = C::COL_DV, COL_DK = C::COL_DK, COL_DQ = C::COL_DQ;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bars->sched_full[s], 1);
      mbar_init(&bars->sched_empty[s], C::SCHED_CONSUMERS + (ROPE ? 2 : 0));
    }
    mbar_init(&bars->clc_bar, 1);
    for (int s = 0; s < C::NQK; ++s) {
      mbar_init(&bars->qk_full[s], 1);
      mbar_init(&bars->qk_empty[s], 1);
      mbar_init(&bars->qk_rot[s], 2);
    }
    for (int s = 0; s < C::NVD; ++s) {
      mbar_init(&bars->vdo_full[s], 1);
      mbar_init(&bars->vdo_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_used, 1);
    mbar_init(&bars->stg_free, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->box_full[b], 128);
      mbar_init(&bars->box_free[b], 1);
    }
    mbar_init(&bars->p_full, 4);
    mbar_init(&bars->ds_full, 4);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->t_free, 4);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const Abort ab{&bars->abort_flag, p.err};

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- loader and scheduler
    // Per tile, in order: QK(i) (its slot was freed by tile i-2) and VdO(i)
    // (free once tile i-1's dV has run), across chunk boundaries.  The block
    // search runs once per pair of blocks, shared by the pair's heads.
    int cached_pair = -1;
    Blk ca{0, 0}, cb{0, 0};
    Locator locate;
    auto rows = [&](int t, Blk& a, Blk& b, int& h) {
      const int pair = t / p.H;
      h = t % p.H;
      if (pair != cached_pair) {
        cached_pair = pair;
        ca = locate(p, 2 * pair);
        cb = locate(p, 2 * pair + 1);
        if (cb.len == 0) cb = ca;
      }
      a = ca;
      b = cb;
    };
    auto load_qk = [&](int i, int t) -> bool {
      const int st = i % C::NQK;
      if (!mbar_wait(&bars->qk_empty[st], ((i / C::NQK) & 1) ^ 1, ab)) return false;
      Blk a, b;
      int h;
      rows(t, a, b, h);
      uint8_t* base = smem + st * 2 * C::TILE;
      mbar_expect_tx(&bars->qk_full[st], 2 * C::TILE);
      load_half<D>(&tm_q, &bars->qk_full[st], base, 0, h, a.row0);
      load_half<D>(&tm_q, &bars->qk_full[st], base, 1, h, b.row0);
      load_half<D>(&tm_k, &bars->qk_full[st], base + C::TILE, 0, h, a.row0);
      load_half<D>(&tm_k, &bars->qk_full[st], base + C::TILE, 1, h, b.row0);
      return true;
    };
    auto load_vdo = [&](int i, int t) -> bool {
      const int sv = i % C::NVD;
      if (!mbar_wait(&bars->vdo_empty[sv], ((i / C::NVD) & 1) ^ 1, ab)) return false;
      Blk a, b;
      int h;
      rows(t, a, b, h);
      uint8_t* base = smem + C::OFF_V + sv * 2 * C::TILE;
      mbar_expect_tx(&bars->vdo_full[sv], 2 * C::TILE);
      load_half<D>(&tm_v, &bars->vdo_full[sv], base, 0, h, a.row0);
      load_half<D>(&tm_v, &bars->vdo_full[sv], base, 1, h, b.row0);
      load_half<D>(&tm_do, &bars->vdo_full[sv], base + C::TILE, 0, h, a.row0);
      load_half<D>(&tm_do, &bars->vdo_full[sv], base + C::TILE, 1, h, b.row0);
      return true;
    };
    int cur = p.use_clc ? static_cast<int>(blockIdx.x) : 0;
    int i = 0;
    for (uint32_t sit = 0;; ++sit) {
      if (!publish(bars, sit, cur, p, ab) || cur < 0) break;
      int tb, te;
      chunk_range(p, cur, &tb, &te);
      bool ok = true;
      for (int t = tb; t < te && ok; ++t, ++i) ok = load_qk(i, t) && load_vdo(i, t);
      if (!ok) break;
      cur = next_entry(bars, sit, p, ab);
      if (cur == -2) break;
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    const uint32_t id_s = idesc_bf16(128, 128, 0, 0);   // S = Q K^T, dP = dO V^T
    const uint32_t id_kv = idesc_bf16(128, D, 1, 1);    // dV = P^T dO, dK = dS^T Q
    const uint32_t id_q = idesc_bf16(128, D, 0, 1);     // dQ = dS K
    const uint32_t sP = smem_u32(smem + C::OFF_PDS), sDS = sP;
    TileCursor cur;
    for (int i = 0;; ++i) {
      if (next_tile(cur, bars, p, ab, false) < 0) break;
      const int st = i % C::NQK, sv = i % C::NVD;
      const uint32_t q = smem_u32(smem + st * 2 * C::TILE), k = q + C::TILE;
      const uint32_t v = smem_u32(smem + C::OFF_V + sv * 2 * C::TILE), dO = v + C::TILE;
      if (!mbar_wait(ROPE ? &bars->qk_rot[st] : &bars->qk_full[st], (i / C::NQK) & 1, ab)) break;
      // S and dP reuse their columns once the softmax warps have read the
      // previous tile's (p_full and ds_full, waited below for that tile); with
      // the accumulators in the same columns, the epilogue must also be done
      if (!C::SPLIT && !mbar_wait(&bars->t_free, (i & 1) ^ 1, ab)) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
        mma_ss(tmem + COL_S, sdesc_sw128(q + off, 16, 1024), sdesc_sw128(k + off, 16, 1024), id_s, kk > 0);
      }
      mma_commit(&bars->s_full);
      if (!mbar_wait(&bars->vdo_full[sv], (i / C::NVD) & 1, ab)) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
        mma_ss(tmem + COL_DP, sdesc_sw128(dO + off, 16, 1024), sdesc_sw128(v + off, 16, 1024), id_s, kk > 0);
      }
      mma_commit(&bars->dp_full);
      // dV = P^T dO: A = P^T (P stored query-major: MN-major), B = dO (MN-major)
      if (!mbar_wait(&bars->p_full, i & 1, ab)) break;
      // separate accumulators: the previous tile's epilogue has read them out
      if (C::SPLIT && !mbar_wait(&bars->t_free, (i & 1) ^ 1, ab)) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tmem + COL_DV, sdesc_sw128(sP + kk * 2048, C::CHUNK, 1024), sdesc_sw128(dO + kk * 2048, C::CHUNK, 1024),
               id_kv, kk > 0);
      mma_commit(&bars->vdo_empty[sv]);  // V and dO are read: the slot may load again
      mma_commit(&bars->p_used);     // P is read: the dS phase may overwrite it
      // dK = dS^T Q, dQ = dS K
      if (!mbar_wait(&bars->ds_full, i & 1, ab)) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tmem + COL_DK, sdesc_sw128(sDS + kk * 2048, C::CHUNK, 1024), sdesc_sw128(q + kk * 2048, C::CHUNK, 1024),
               id_kv, kk > 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
        mma_ss(tmem + COL_DQ, sdesc_sw128(sDS + off, 16, 1024), sdesc_sw128(k + kk * 2048, C::CHUNK, 1024), id_q,
               kk > 0);
      }
      mma_commit(&bars->acc_full);
      mma_commit(&bars->qk_empty[st]);
    }
    mma_commit(&bars->drain);
    const uint64_t tw = global_timer_ns();
    while (!mbar_try_wait(&bars->drain, 0) && global_timer_ns() - tw < kWaitTimeoutNs) {
    }
  } else if (ROPE && (warp == 2 || warp == 3)) {
    // ---------------------------------------------------------------- rotation (rotary variant)
    rope_role<D, C::NQK, 64, D == 128 ? 4 : 2>(p, bars, smem, C::TILE, warp - 2, 0, ab);
  } else if (warp >= 4 && warp < 8) {
    // ---------------------------------------------------------------- softmax, dS (and the epilogue at D = 128)
    const int r = threadIdx.x & 127;
    const int half = r >> 6, rr = r & 63;
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint8_t* sP = smem + C::OFF_PDS;
    uint8_t* sDS = sP;  // the same buffer: dS goes in once the dV GEMM has read P
    const float sl2 = p.scale_log2;
    const uint32_t zero[4] = {0u, 0u, 0u, 0u};
    uint32_t stg_free_ph = 0;
    uint32_t box_full_ph[2] = {0, 0}, box_free_ph[2] = {0, 0};
    TileCursor cur;
    Locator locate;
    for (int i = 0;; ++i) {
      const int t = next_tile(cur, bars, p, ab, true);
      if (t == -2) goto done;
      if (t < 0) break;
      const int pair = t / p.H, h = t % p.H;
      const Blk blk = locate(p, 2 * pair + half);
      if (!mbar_wait(&bars->s_full, i & 1, ab)) goto done;
      tc_fence_after();
      float pr[64];
      {
        uint32_t sr[64];
        tmem_ld32(tmem + lane_addr + COL_S + 64 * half, sr);
        tmem_ld32(tmem + lane_addr + COL_S + 64 * half + 32, sr + 32);
        tmem_wait_ld();
        reg_fence<64>(sr);
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          pr[c] = c < blk.len ? __uint_as_float(sr[c]) * sl2 : -INFINITY;
          mx = fmaxf(mx, pr[c]);
        }
        if (blk.len == 0) mx = 0.f;
        float l = 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          pr[c] = ex2(pr[c] - mx);
          l += pr[c];
        }
        const float inv_l = (rr < blk.len && l > 0.f) ? 1.0f / l : 0.f;  // rows past the block: P = 0
#pragma unroll
        for (int c = 0; c < 64; ++c) pr[c] *= inv_l;
      }
      // P row into shared memory (zeros in the other block's columns); with the
      // separate epilogue the buffer still holds the previous tile's dS until its
      // dK and dQ GEMMs are done
      if (C::SPLIT && i > 0 && !mbar_wait(&bars->acc_full, (i - 1) & 1, ab)) goto done;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = pack_bf16(pr[8 * j + 2 * e], pr[8 * j + 2 * e + 1]);
        st_row_piece(sP, r, half, j, w);
        st_row_piece(sP, r, 1 - half, j, zero);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full);
      // dS = P o (dP - Di), Di = rowsum(P o dP) over this block's keys
      if (!mbar_wait(&bars->dp_full, i & 1, ab)) goto done;
      tc_fence_after();
      {
        uint32_t dr[64];
        tmem_ld32(tmem + lane_addr + COL_DP + 64 * half, dr);
        tmem_ld32(tmem + lane_addr + COL_DP + 64 * half + 32, dr + 32);
        tmem_wait_ld();
        reg_fence<64>(dr);
        float di = 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c) di = fmaf(pr[c], __uint_as_float(dr[c]), di);
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2)
          w[c / 2] = pack_bf16(pr[c] * (__uint_as_float(dr[c]) - di), pr[c + 1] * (__uint_as_float(dr[c + 1]) - di));
        if (!mbar_wait(&bars->p_used, i & 1, ab)) goto done;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          st_row_piece(sDS, r, half, j, w + 4 * j);
          st_row_piece(sDS, r, 1 - half, j, zero);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->ds_full);
      if constexpr (D == 128) {
        // epilogue: row r is query r for dQ and key r for dK, dV (same block, same token).
        // Each result is staged as bf16 rows in the P/dS buffer (free once dK and dQ
        // have read dS) and written by TMA, one 64-row half at a time; a half whose
        // block is shorter than 64 rows is written row by row instead, so no rows
        // of the next block are touched.
        // thread 128 (row 0, block a) issues the stores; it also needs block b
        const Blk blk_a = blk, blk_b = threadIdx.x == 128 ? locate(p, 2 * pair + 1) : blk;
        // rotary: the table row of this thread's token (64 pairs), loaded while
        // the tile's last GEMMs run; dQ and dK share it
        uint4 tab[ROPE ? D / 8 : 1];
        if constexpr (ROPE) {
          const uint4* e = reinterpret_cast<const uint4*>(p.rope_tab + static_cast<size_t>(blk.pos0 + rr) * (D / 2));
#pragma unroll
          for (int j = 0; j < D / 8; ++j) tab[j] = rr < blk.len ? __ldg(e + j) : make_uint4(0u, 0u, 0u, 0u);
        }
        if (!mbar_wait(&bars->acc_full, i & 1, ab)) goto done;
        tc_fence_after();
        {
          const bool valid = rr < blk.len;
          const bool full_half = blk.len == kBlk;
          const size_t row = (static_cast<size_t>(blk.row0 + rr) * p.H + h) * D;
          {
            // dQ, dK, dV one 64-column box at a time through the two halves of
            // the staging buffer: the rows of one box are written while TMA still
            // reads the other.  Rotary: dQ and dK are gradients with respect to
            // the rotated rows, so the whole fp32 row goes back through the
            // transposed rotation (pairs (i, i + D/2)) into registers first, then
            // its two boxes are staged in turn.
            uint32_t wrow[ROPE ? D / 2 : 1];  // rotary: the row's bf16 pairs
  #pragma unroll 1
            for (int which = 0; which < 3; ++which) {
              const uint32_t col = which == 0 ? COL_S : (which == 1 ? COL_DP : COL_DV);
              const float mul = which == 2 ? 1.0f : p.scale;
              const CUtensorMap* tm_out = which == 0 ? &tm_dq : (which == 1 ? &tm_dk : &tm_dv);
              __nv_bfloat16* dst = (which == 0 ? p.dq : (which == 1 ? p.dk : p.dv)) + row;
              const bool rotated = ROPE && which < 2;
              if constexpr (ROPE) {
                if (rotated) {
                  const uint64_t sc = f32x2(mul, mul);
  #pragma unroll
                  for (int r2 = 0; r2 < 2; ++r2) {
                    uint32_t vx[32], vy[32];
                    tmem_ld32(tmem + lane_addr + col + 32 * r2, vx);
                    tmem_ld32(tmem + lane_addr + col + D / 2 + 32 * r2, vy);
                    tmem_wait_ld();
                    reg_fence<32>(vx);
                    reg_fence<32>(vy);
  #pragma unroll
                    for (int e = 0; e < 16; ++e) {
                      // cos and sin of pairs (32 r2 + 2e, +1), times the softmax scale
                      const uint4& tq = tab[8 * r2 + e / 2];
                      const uint64_t c = fmul2(h2_to_f32x2(e & 1 ? tq.z : tq.x), sc);
                      const uint64_t sn = fmul2(h2_to_f32x2(e & 1 ? tq.w : tq.y), sc);
                      uint64_t uo, vo;
                      rot2<true>(f32x2(__uint_as_float(vx[2 * e]), __uint_as_float(vx[2 * e + 1])),
                                 f32x2(__uint_as_float(vy[2 * e]), __uint_as_float(vy[2 * e + 1])), c, sn, uo, vo);
                      wrow[16 * r2 + e] = f32x2_to_bf16x2(uo);
                      wrow[D / 4 + 16 * r2 + e] = f32x2_to_bf16x2(vo);
                    }
                  }
                }
              }
  #pragma unroll
              for (int box = 0; box < 2; ++box) {
              const int s = 2 * which + box;
              if (s >= 2) {  // the box's previous rows (two stages back) have been read out
                if (threadIdx.x == 128) {
                  bulk_wait_read_all_but_newest();
                  mbar_arrive(&bars->box_free[box]);
                }
                if (!mbar_wait(&bars->box_free[box], box_free_ph[box], ab)) goto done;
                box_free_ph[box] ^= 1;
              }
  #pragma unroll
              for (int c = 64 * box; c < 64 * box + 64; c += 32) {
                uint32_t w[16];
                if (rotated) {
  #pragma unroll
                  for (int e = 0; e < 16; ++e) w[e] = wrow[(ROPE ? c / 2 : 0) + e];
                } else {
                  uint32_t v[32];
                  tmem_ld32(tmem + lane_addr + col + c, v);
                  tmem_wait_ld();
                  reg_fence<32>(v);
  #pragma unroll
                  for (int e = 0; e < 16; ++e)
                    w[e] = pack_bf16(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
                }
  #pragma unroll
                for (int e = 0; e < 4; ++e) st_row_piece(sP, r, box, (c % 64) / 8 + e, w + 4 * e);
                if (valid && !full_half) {
  #pragma unroll
                  for (int e = 0; e < 4; ++e)
                    st_global_v4(dst + c + 8 * e, w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                }
              }
              if (s == 5) {  // every accumulator has been read: TMEM is free
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->t_free);
              }
              fence_proxy_async_smem();
              mbar_arrive(&bars->box_full[box]);
              if (!mbar_wait(&bars->box_full[box], box_full_ph[box], ab)) goto done;
              box_full_ph[box] ^= 1;
              if (threadIdx.x == 128) {
  #pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                  const Blk bk = hf == 0 ? blk_a : blk_b;
                  if (bk.len == kBlk)
                    tma_store_2d(tm_out, smem + C::OFF_PDS + box * 16384 + hf * 8192, h * D + 64 * box, bk.row0);
                }
                bulk_commit_group();
              }
              }
            }
          }
          // the next tile's P goes into the same buffer: wait for the last boxes
          if (threadIdx.x == 128) {
            bulk_wait_read_all();
            mbar_arrive(&bars->stg_free);
          }
          if (!mbar_wait(&bars->stg_free, stg_free_ph, ab)) goto done;
          stg_free_ph ^= 1;
        }
      }
    }
    if (threadIdx.x == 128) bulk_wait_all();  // every store has landed before the CTA exits
  } else if (C::SPLIT && warp >= 8) {
    // ---------------------------------------------------------------- epilogue (D = 64)
    // Row r is query r for dQ and key r for dK, dV (same block, same token); each
    // thread writes its rows directly (at this head size the staged path measured
    // slower), while the softmax warps already work on the next tile.
    const int r = threadIdx.x & 127;
    const int half = r >> 6, rr = r & 63;
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    TileCursor cur;
    Locator locate;
    for (int i = 0;; ++i) {
      const int t = next_tile(cur, bars, p, ab, true);
      if (t == -2) goto done;
      if (t < 0) break;
      const int pair = t / p.H, h = t % p.H;
      const Blk blk = locate(p, 2 * pair + half);
      const bool valid = rr < blk.len;
      // rotary: the table row of this thread's token (32 pairs), loaded while
      // the tile's GEMMs finish; dQ and dK share it
      uint4 tab[ROPE ? D / 8 : 1];
      if constexpr (ROPE && D == 64) {
        if (valid) {
          const uint4* e = reinterpret_cast<const uint4*>(p.rope_tab + static_cast<size_t>(blk.pos0 + rr) * (D / 2));
#pragma unroll
          for (int j = 0; j < D / 8; ++j) tab[j] = __ldg(e + j);
        }
      }
      if (!mbar_wait(&bars->acc_full, i & 1, ab)) goto done;
      tc_fence_after();
      {
        const size_t row = (static_cast<size_t>(blk.row0 + rr) * p.H + h) * D;
#pragma unroll 1
        for (int which = 0; which < 3; ++which) {
          const uint32_t col = which == 0 ? COL_DQ : (which == 1 ? COL_DK : COL_DV);
          const float mul = which == 2 ? 1.0f : p.scale;
          __nv_bfloat16* dst = (which == 0 ? p.dq : (which == 1 ? p.dk : p.dv)) + row;
          if constexpr (ROPE && D == 64) {
            if (which < 2) {
              // dQ and dK are gradients with respect to the rotated rows: the
              // transposed rotation of the whole fp32 row, pairs (i, i + D/2),
              // (g_i, g_i') -> (g_i c + g_i' s, g_i' c - g_i s), rounded once
              const uint64_t sc = f32x2(mul, mul);
#pragma unroll
              for (int r2 = 0; r2 < 2; ++r2) {  // pairs [16 r2, 16 r2 + 16)
                uint32_t vx[16], vy[16];
                tmem_ld16(tmem + lane_addr + col + 16 * r2, vx);
                tmem_ld16(tmem + lane_addr + col + D / 2 + 16 * r2, vy);
                tmem_wait_ld();
                reg_fence<16>(vx);
                reg_fence<16>(vy);
                if (valid) {
                  uint32_t wx[8], wy[8];
#pragma unroll
                  for (int e = 0; e < 8; ++e) {
                    // cos and sin of pairs (16 r2 + 2e, +1), times the softmax scale
                    const uint4& tq = tab[4 * r2 + e / 2];
                    const uint64_t c = fmul2(h2_to_f32x2(e & 1 ? tq.z : tq.x), sc);
                    const uint64_t sn = fmul2(h2_to_f32x2(e & 1 ? tq.w : tq.y), sc);
                    uint64_t uo, vo;
                    rot2<true>(f32x2(__uint_as_float(vx[2 * e]), __uint_as_float(vx[2 * e + 1])),
                               f32x2(__uint_as_float(vy[2 * e]), __uint_as_float(vy[2 * e + 1])), c, sn, uo, vo);
                    wx[e] = f32x2_to_bf16x2(uo);
                    wy[e] = f32x2_to_bf16x2(vo);
                  }
#pragma unroll
                  for (int e = 0; e < 2; ++e) {
                    st_global_v4(dst + 16 * r2 + 8 * e, wx[4 * e], wx[4 * e + 1], wx[4 * e + 2], wx[4 * e + 3]);
                    st_global_v4(dst + D / 2 + 16 * r2 + 8 * e, wy[4 * e], wy[4 * e + 1], wy[4 * e + 2],
                                 wy[4 * e + 3]);
                  }
                }
              }
              continue;
            }
          }
          // columns c..c+31 of the result row, as fp32, stored
          auto put = [&](int c, const float* f) {
            if (!valid) return;
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) w[e] = pack_bf16(f[2 * e], f[2 * e + 1]);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              st_global_v4(dst + c + 8 * e, w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
          };
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_addr + col + c, v);
            tmem_wait_ld();
            reg_fence<32>(v);
            float f[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(v[e]) * mul;
            put(c, f);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->t_free);
      }
    }
  }
done:
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool ROPE>
int launch_fwd_impl(const BlockArgs& a) {
  using C = FwdCfg<D>;
  static_assert(C::SMEM <= 232448, "shared memory budget");
  CUtensorMap tq, tk, tv;
  const uint64_t inner = static_cast<uint64_t>(a.H) * D;
  int st = make_map_2d(&tq, a.q, inner, a.rows, 64, kBlk);
  if (st == JFA_OK) st = make_map_2d(&tk, a.k, inner, a.rows, 64, kBlk);
  if (st == JFA_OK) st = make_map_2d(&tv, a.v, inner, a.rows, 64, kBlk);
  if (st != JFA_OK) return st;
  static PerDeviceOnce setup;  // per instantiation
  st = setup.run([]() -> int {
    return cudaFuncSetAttribute(block_fwd_kernel<D, ROPE>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) ==
                   cudaSuccess
               ? JFA_OK
               : JFA_ERR_CUDA;
  });
  if (st != JFA_OK) return st;
  Params p{};
  p.offsets = a.offsets_dev;
  p.bpb = a.bpb;
  p.prog_start = a.prog_start;
  p.err = a.err;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.batch = a.batch;
  p.H = a.H;
  p.n_blocks = a.n_blocks;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.use_clc = a.use_clc;
  p.chunk = a.chunk;
  p.n_tiles = a.n_tiles;
  p.n_chunks = a.n_chunks;
  p.rope_tab = a.rope_tab;
  ProfileScope prof(kKindBlockFwd, a.stream);
  block_fwd_kernel<D, ROPE><<<a.use_clc ? a.n_chunks : a.n_prog, ROPE ? 512 : 384, C::SMEM, a.stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

template <int D, bool ROPE>
int launch_bwd_impl(const BlockArgs& a) {
  using C = BwdCfg<D>;
  static_assert(C::SMEM <= 232448, "shared memory budget");
  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
  const uint64_t inner = static_cast<uint64_t>(a.H) * D;
  int st = make_map_2d(&tq, a.q, inner, a.rows, 64, kBlk);
  if (st == JFA_OK) st = make_map_2d(&tk, a.k, inner, a.rows, 64, kBlk);
  if (st == JFA_OK) st = make_map_2d(&tv, a.v, inner, a.rows, 64, kBlk);
  if (st == JFA_OK) st = make_map_2d(&tdo, a.dout, inner, a.rows, 64, kBlk);
  if (st == JFA_OK) st = make_map_2d(&tdq, a.dq, inner, a.rows, 64, kBlk);
  if (st == JFA_OK) st = make_map_2d(&tdk, a.dk, inner, a.rows, 64, kBlk);
  if (st == JFA_OK) st = make_map_2d(&tdv, a.dv, inner, a.rows, 64, kBlk);
  if (st != JFA_OK) return st;
  static PerDeviceOnce setup;  // per instantiation
  st = setup.run([]() -> int {
    return cudaFuncSetAttribute(block_bwd_kernel<D, ROPE>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) ==
                   cudaSuccess
               ? JFA_OK
               : JFA_ERR_CUDA;
  });
  if (st != JFA_OK) return st;
  Params p{};
  p.offsets = a.offsets_dev;
  p.bpb = a.bpb;
  p.prog_start = a.prog_start;
  p.err = a.err;
  p.dq = static_cast<__nv_bfloat16*>(a.dq);
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.batch = a.batch;
  p.H = a.H;
  p.n_blocks = a.n_blocks;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.use_clc = a.use_clc;
  p.chunk = a.chunk;
  p.n_tiles = a.n_tiles;
  p.n_chunks = a.n_chunks;
  p.rope_tab = a.rope_tab;
  ProfileScope prof(kKindBlockBwd, a.stream);
  block_bwd_kernel<D, ROPE><<<a.use_clc ? a.n_chunks : a.n_prog, C::THREADS, C::SMEM, a.stream>>>(
      tq, tk, tv, tdo, tdq, tdk, tdv, p);
  return cudaGetLastError() == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

}  // namespace blk

int launch_block_fwd(const BlockArgs& a) {
  if (a.rope_tab != nullptr)
    return a.D == 128 ? blk::launch_fwd_impl<128, true>(a) : blk::launch_fwd_impl<64, true>(a);
  return a.D == 128 ? blk::launch_fwd_impl<128, false>(a) : blk::launch_fwd_impl<64, false>(a);
}
int launch_block_bwd(const BlockArgs& a) {
  if (a.rope_tab != nullptr)
    return a.D == 128 ? blk::launch_bwd_impl<128, true>(a) : blk::launch_bwd_impl<64, true>(a);
  return a.D == 128 ? blk::launch_bwd_impl<128, false>(a) : blk::launch_bwd_impl<64, false>(a);
}

}  // namespace jfa
