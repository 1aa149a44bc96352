// bwd.cu -- jagged flash-attention backward for sm_103a.
//
// What it computes, per (sequence, head), given Q, K, V, O, dO and the forward's
// log-sum-exp L ("TLX Block Attention", section 4; the aixai.ru summary counts
// five GEMMs per K/V block, "Paired CTAs"):
//   P  = exp(scale Q K^T - L)            (recomputed, no stored P)
//   dV = P^T dO,  dP = dO V^T,  Di = rowsum(dO o O),  dS = P o (dP - Di)
//   dQ = scale dS K,  dK = scale dS^T Q
// Broadcast-Q sums dQ of the shared Q over every sequence.  With grouped-query
// attention (G = H / Hkv query heads per K/V head) dK and dV of a K/V head sum
// the contributions of all G query heads of its group.
//
// Kernels, in launch order:
//   prep_kernel   Di = rowsum(dO o O) and L * log2(e) per (row, head); zeroes the
//                 fp32 dQ accumulator
//   bwd_kernel    persistent, one CTA per SM, one work unit = one valid block of
//                 128 keys of one (sequence, K/V head); it loops over the query
//                 heads of the head's group and, per head, the 128-row query
//                 tiles that attend to those keys, keeps dK and dV in TMEM and
//                 adds each tile's dQ into an fp32 accumulator
//   dq_convert    dQ = scale * accumulator -> bf16
//
// bwd_kernel roles (warp specialisation as in the aixai.ru summary, "Framework",
// including the dedicated dQ-reduction role):
//   warps 0-3 / 4-7  one thread per key (TMEM lane); warpgroup w handles query
//                    columns [64w, 64w+64): P^T (bf16, into TMEM) and dS^T (bf16,
//                    into swizzled shared memory)
//   warps 8-11       dQ reduction and dK/dV epilogue: one thread per TMEM lane; at
//                    the end of a unit it writes dV and dK (before that tile's dQ,
//                    so the next unit's dV/dK MMAs can start); per tile it reads dQ,
//                    releases TMEM as soon as the whole row is in registers, stages
//                    the tile in shared memory and reduce-adds it into the fp32
//                    accumulator with TMA (aixai.ru summary, "dQ epilogue": staged
//                    writeback and early TMEM release)
//   warp 12          tcgen05 MMA issuer
//   warp 13          loader and scheduler: publishes each unit index to the other
//                    roles through a 4-slot ring (the CTA's slice of the static
//                    plan, or under Cluster Launch Control its own unit and then
//                    those of CTAs whose launch it cancels); K, V by TMA once per
//                    unit; per query tile Q by TMA into a 2-deep ring (with L, Di
//                    into shared memory) and dO into a single buffer (dV, its last
//                    reader, runs early in each tile)
// TMEM: two 128-column regions that S^T and dP^T swap every tile (P^T overwrites
// columns 0-31 and 64-95 of S^T's region; that tile's dQ then reuses the region),
// dV [256,256+D), dK [256+D, 256+2D).
// Per tile the tensor core runs dP^T = V dO^T, dV += P^T dO, dQ = dS K, the next
// tile's S^T = K Q^T, then dK += dS^T Q: the next tile's P phase overlaps dK and
// the next dP^T, and no S^T waits for the dQ drain.
// Masks: keys past the sequence end and query rows past it are zeroed per thread
// (a key flag and L = +inf), so only the causal diagonal tile -- or, under a
// sliding window, a tile that straddles the window's edge -- needs an
// element-wise mask, and it is peeled into its own code path.  Under a window
// a unit visits only the query tiles that see its keys.
#include <algorithm>
#include <type_traits>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "bwd.h"
#include "host.h"
#include "profile.h"
#include "ptx.cuh"

namespace jfa {
namespace bwd {

constexpr int BQ = 128;  // query rows per tile
constexpr int BK = 128;  // keys per unit
constexpr int kThreads = 512;
// Registers per thread after setmaxnreg: the two P/dS warpgroups, the dQ/dK/dV
// drain warpgroup, the MMA/loader warpgroup.  The sum must not exceed the
// launch allocation (128 per thread at 512 threads); the launcher checks the
// compiled count.
constexpr int kRegPds = 128, kRegDrain = 160, kRegIssue = 96;
constexpr int kRegTotal = 2 * 128 * kRegPds + 128 * kRegDrain + 128 * kRegIssue;
static_assert(kRegTotal <= kThreads * 128, "register split exceeds the launch allocation");
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct Cfg {
  static constexpr int TILE = 128 * D * 2;      // one 128-row bf16 tile
  static constexpr int CHUNK = 128 * 128;        // one 64-column swizzle box (bytes)
  static constexpr int NQS = 2;                  // Q/dO ring depth
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_Q = OFF_V + TILE;                 // NQS x Q
  static constexpr int OFF_DO = OFF_Q + NQS * TILE;          // one dO tile: dV, its last reader,
                                                             // runs early in a tile, so one buffer suffices
  static constexpr int OFF_DS = OFF_DO + TILE;               // dS^T [128 keys][128 queries] bf16
  static constexpr int OFF_STG = OFF_DS + 128 * 128 * 2;     // dQ staging: two 32-column fp32 boxes
  static constexpr int OFF_BAR = OFF_STG + 2 * 128 * 128;
  static constexpr int OFF_LD = OFF_BAR + 384;                    // per-stage L and Di, 128 floats each
  static constexpr int SMEM_BYTES = OFF_LD + NQS * 1024;
  // No alignment slack: at head_dim 128 this is within 1 KB of the 227 KB limit.
  // The kernel checks that dynamic shared memory starts 1024-byte aligned.
  static constexpr int SMEM_ALLOC = SMEM_BYTES;
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
  static constexpr uint32_t COL_DV = 256;
  static constexpr uint32_t COL_DK = 256 + D;
};

struct Params {
  const int4* units;
  const int32_t* cta_start;
  const int32_t* offsets;
  const float* lse2;   // [H, o_rows]  L * log2(e)
  const float* di;     // [H, o_rows]
  float* dq_acc;       // [q_rows, H, D]
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int* err;
  int H, Hkv, G, nq, o_rows;  // G = H / Hkv query heads per K/V head
  float scale, scale_log2;
  int use_clc;  // 1: one CTA per unit in cost order, CTAs take over units of CTAs not yet launched
  int n_units;
  int win_left, win_right;  // sliding window (kMaskWindow): keys [row - left, row + right], -1 = open
};

struct Unit {
  int b, h, n;         // h: the K/V head; its query heads are h*G .. h*G+G-1
  int kv0, L;          // first key row of the sequence, its length
  int rows;            // query rows (L, or nq in broadcast mode)
  int i0, i1;          // query tiles [i0, i1)
  int q_base, o_base;  // row of query 0 in q / in o
};

template <int MASK>
__device__ __forceinline__ Unit decode(const Params& p, int idx) {
  const int4 e = p.units[idx];
  Unit u;
  u.b = e.x;
  u.h = e.y;
  u.n = e.z;
  u.kv0 = p.offsets[u.b];
  u.L = e.w;  // the sequence length (the host wrote it into the entry)
  if (p.nq > 0) {
    u.rows = p.nq;
    u.q_base = 0;
    u.o_base = u.b * p.nq;
  } else {
    u.rows = u.L;
    u.q_base = u.kv0;
    u.o_base = u.kv0;
  }
  if (MASK == kMaskWindow) {  // the query rows that see some key of this block
    const int k_last = min(BK * (u.n + 1), u.L) - 1;
    const int lo = p.win_right < 0 ? 0 : max(0, BK * u.n - p.win_right);
    const int hi = p.win_left < 0 ? u.rows : min(u.rows, k_last + p.win_left + 1);
    u.i0 = lo / BQ;
    u.i1 = (hi + BQ - 1) / BQ;
  } else {
    u.i0 = MASK == kMaskCausal ? u.n : 0;
    u.i1 = (u.rows + BQ - 1) / BQ;
  }
  return u;
}

// Whether query tile i sees some but not all of the keys of block n (so its P
// needs the element mask): the causal diagonal tile, or a tile across a
// window edge.
template <int MASK>
__device__ __forceinline__ bool edge_tile(const Params& p, int i, int n) {
  if (MASK == kMaskCausal) return i == n;
  if (MASK == kMaskWindow)
    return (p.win_left >= 0 && BK * n < BQ * i + BQ - 1 - p.win_left) ||
           (p.win_right >= 0 && BK * n + BK - 1 > BQ * i + p.win_right);
  return false;
}

// TMEM column of this tile's S^T (and later of its dQ); dP^T takes the other
// 128-column region.  The two swap every tile.
__device__ __forceinline__ uint32_t region_s(uint32_t tile_counter) { return (tile_counter & 1) ? 128u : 0u; }

struct Bars {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[2], q_empty[2], do_full, do_empty;
  uint64_t s_full, dp_full, p_full, ds_full, ds_empty, dq_full, dq_empty, dkv_full, dkv_empty;
  uint64_t stg_full[2], stg_free[2];  // dQ staging slots: rows written by the 128 drain threads / read out by TMA
  uint64_t kvst_full, kvst_free;      // the same buffer holding a bf16 dK or dV tile for a TMA store
  uint64_t drain;
  // unit schedule: the loader publishes each unit index (or -1 at the end) to
  // the other roles through this ring
  uint64_t sched_full[4], sched_empty[4], clc_bar;
  int4 clc_resp;
  int sched_unit[4];
  uint32_t tmem_base;
  int abort_flag;
};

constexpr int kSchedConsumers = 13;  // 8 P/dS warps + 4 drain warps + the MMA thread

// FINE: the broadcast-Q instantiation, whose dK/dV epilogue is pipelined per box
template <int D, int MASK, bool FINE = false>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
               const __grid_constant__ CUtensorMap tm_dv, const Params p) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023) != 0) {  // the layout below needs 1024-byte alignment
    if (threadIdx.x == 0 && p.err) atomicCAS(p.err, 0, kDevMisaligned);
    return;
  }
  uint8_t* smem = smem_raw;
  Bars* bars = reinterpret_cast<Bars*>(smem + C::OFF_BAR);
  static_assert(sizeof(Bars) <= 384, "barrier block");
  float* s_lse = reinterpret_cast<float*>(smem + C::OFF_LD);  // [NQS][128]
  float* s_di = s_lse + C::NQS * 128;                          // [NQS][128]

  const int warp = warp_id();
  const int lane = lane_id();
  const int u_begin = p.use_clc ? 0 : p.cta_start[blockIdx.x];
  const int u_end = p.use_clc ? 0 : p.cta_start[blockIdx.x + 1];

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->q_full[s], 32);
      mbar_init(&bars->q_empty[s], 1);
    }
    mbar_init(&bars->do_full, 1);
    mbar_init(&bars->do_empty, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, 8);
    mbar_init(&bars->ds_full, 8);
    mbar_init(&bars->ds_empty, 1);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_empty, 4);
    mbar_init(&bars->dkv_full, 1);
    mbar_init(&bars->dkv_empty, 4);
    mbar_init(&bars->kvst_full, 128);
    mbar_init(&bars->kvst_free, 1);
    for (int s2 = 0; s2 < 2; ++s2) {
      mbar_init(&bars->stg_full[s2], 128);
      mbar_init(&bars->stg_free[s2], 1);
    }
    mbar_init(&bars->drain, 1);
    for (int s3 = 0; s3 < 4; ++s3) {
      mbar_init(&bars->sched_full[s3], 1);
      mbar_init(&bars->sched_empty[s3], kSchedConsumers);
    }
    mbar_init(&bars->clc_bar, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 12) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const Abort ab{&bars->abort_flag, p.err};

  if (warp < 8) {
    // -------------------------------------------------------- P^T and dS^T
    // register split 128 / 128 / 160 / 96 over the four warpgroups (65,536 total)
    setmaxnreg_inc<kRegPds>();
    const int wg = warp >> 2;              // query half
    const int k = threadIdx.x & 127;       // key row == TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint8_t* sDS = smem + C::OFF_DS + wg * C::CHUNK + k * 128;  // row k of this half's box
    const float sl2 = p.scale_log2;
    uint32_t ph = 0, ds_ph = 0, q_it = 0;
    for (uint32_t it = 0;; ++it) {
      const int ui = sched_pop(bars, it, ab, true);
      if (ui == -2) goto done;
      if (ui < 0) break;
      const Unit u = decode<MASK>(p, ui);
      const bool key_ok = BK * u.n + k < u.L;
      const bool all_keys_ok = __all_sync(0xffffffffu, key_ok);  // the same in the whole warp
      for (int hg = 0; hg < p.G; ++hg)
      for (int i = u.i0; i < u.i1; ++i, ++q_it) {
        const int st = q_it & 1;
        const float* lse_s = s_lse + st * 128 + 64 * wg;
        const float* di_s = s_di + st * 128 + 64 * wg;
        // S^T and dP^T swap TMEM regions every tile (see the MMA issuer)
        const uint32_t rs = region_s(q_it), rd = 128 - rs;
        const uint32_t tS = tmem + lane_addr + rs + 64 * wg;   // S^T columns of this half
        const uint32_t tP = tS;                                // P^T packed (32 columns)
        const uint32_t tDP = tmem + lane_addr + rd + 64 * wg;
        if (!mbar_wait(&bars->s_full, ph, ab)) goto done;
        tc_fence_after();
        const bool diag = edge_tile<MASK>(p, i, u.n);
        // P^T first: the dV MMA can start while dS^T is being formed.  Only the
        // causal diagonal tile carries the element mask, and only warps with keys
        // past the sequence end the key select (both choices are the same for the
        // whole warp, as the TMEM accesses need).
        float pf[64];
        const int d_base = BQ * (i - u.n) - k;  // query position - key position at column 0
        auto p_phase = [&](auto diag_tile, auto key_mask) {
#pragma unroll
          for (int pass = 0; pass < 2; ++pass) {
            uint32_t sr[32];
            tmem_ld32(tS + 32 * pass, sr);
            tmem_wait_ld();
            reg_fence<32>(sr);
            uint32_t pw[16];
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
              const float4 l4 = *reinterpret_cast<const float4*>(lse_s + 32 * pass + c);
              const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float pe = ex2(fmaf(__uint_as_float(sr[c + e]), sl2, -lv[e]));
                if constexpr (decltype(diag_tile)::value) {
                  if (MASK == kMaskCausal) {
                    if ((64 * wg + 32 * pass + c + e) < k) pe = 0.f;
                  } else {  // query minus key position against the window's bounds
                    const int dq_k = d_base + 64 * wg + 32 * pass + c + e;
                    if ((p.win_left >= 0 && dq_k > p.win_left) || (p.win_right >= 0 && -dq_k > p.win_right))
                      pe = 0.f;
                  }
                }
                if constexpr (decltype(key_mask)::value) pe = key_ok ? pe : 0.f;
                pf[32 * pass + c + e] = pe;
              }
              pw[c / 2] = pack_bf16(pf[32 * pass + c], pf[32 * pass + c + 1]);
              pw[c / 2 + 1] = pack_bf16(pf[32 * pass + c + 2], pf[32 * pass + c + 3]);
            }
            tmem_st16(tP + 16 * pass, pw);
          }
        };
        if (diag)
          p_phase(std::true_type{}, std::true_type{});
        else if (!all_keys_ok)  // a tail block: some keys of this warp lie past the sequence end
          p_phase(std::false_type{}, std::true_type{});
        else
          p_phase(std::false_type{}, std::false_type{});
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full);
        // dS^T = P^T o (dP^T - Di) into shared memory, once the previous tile's
        // dK/dQ MMAs have read it (they were issued before this tile's S^T, so
        // this rarely waits)
        if (!mbar_wait(&bars->ds_empty, ds_ph ^ 1, ab)) goto done;
        ds_ph ^= 1;
        if (!mbar_wait(&bars->dp_full, ph, ab)) goto done;
        ph ^= 1;
        tc_fence_after();
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
          uint32_t dr[32];
          tmem_ld32(tDP + 32 * pass, dr);
          tmem_wait_ld();
          reg_fence<32>(dr);
          uint32_t dsw[16];
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            const float4 d4 = *reinterpret_cast<const float4*>(di_s + 32 * pass + c);
            const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
            float dsv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) dsv[e] = pf[32 * pass + c + e] * (__uint_as_float(dr[c + e]) - dv[e]);
            dsw[c / 2] = pack_bf16(dsv[0], dsv[1]);
            dsw[c / 2 + 1] = pack_bf16(dsv[2], dsv[3]);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int chunk = 4 * pass + j;
            const uint32_t addr = smem_u32(sDS + ((chunk ^ (k & 7)) << 4));
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(dsw[4 * j]),
                         "r"(dsw[4 * j + 1]), "r"(dsw[4 * j + 2]), "r"(dsw[4 * j + 3])
                         : "memory");
          }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->ds_full);
      }
    }
  } else if (warp < 12) {
    // -------------------------------------------------------- dQ reduction
    setmaxnreg_inc<kRegDrain>();
    const int r = threadIdx.x & 127;
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t ph = 0, q_it = 0, dkv_ph = 0, kvst_full_ph = 0, kvst_free_ph = 0;
    for (uint32_t it = 0;; ++it) {
      const int ui = sched_pop(bars, it, ab, true);
      if (ui == -2) goto done;
      if (ui < 0) break;
      const Unit u = decode<MASK>(p, ui);
      for (int hg = 0; hg < p.G; ++hg)
      for (int i = u.i0; i < u.i1; ++i, ++q_it) {
        const uint32_t tQ = tmem + lane_addr + region_s(q_it);  // dQ sits where this tile's S^T was
        if (hg + 1 == p.G && i + 1 == u.i1) {
          // unit done: dV and dK leave TMEM first (the next unit's first dV/dK
          // MMAs wait for them); one thread per key row
          if (!mbar_wait(&bars->dkv_full, dkv_ph, ab)) goto done;
          dkv_ph ^= 1;
          tc_fence_after();
          // A block of 128 valid keys goes out through the staging buffer and TMA
          // stores (one warp store instruction would otherwise touch 32 rows); a
          // shorter tail block is written row by row, so the next sequence's rows
          // are untouched.  The buffer is taken over from the dQ reduction once its
          // boxes have been read.  Causal attention keeps the row stores: its query
          // loads are DRAM-heavy and the stores' TMA traffic measured slower there.
          const bool full_blk = MASK == kMaskNone && BK * (u.n + 1) <= u.L;
          const bool key_ok = BK * u.n + r < u.L;
          const size_t row = (static_cast<size_t>(u.kv0 + BK * u.n + r) * p.Hkv + u.h) * D;
          const uint32_t stage32 = smem_u32(smem + C::OFF_STG);
          // broadcast-Q (two query tiles per unit): the drain is mostly this
          // epilogue, so dV, then dK go one 64-column box per stage through the
          // two 16 KB slots in turn, the rows of one stage written while TMA still
          // reads the previous one (backward call 487 -> 455 us); self-attention
          // units keep one hand-off per tensor, as the finer one measured slower
          // there (jagged 648 -> 653 us; with both paths in one kernel, 661 us)
          const bool fine = FINE && full_blk;
          if (fine) {
            constexpr int NBOX = D / 64;
#pragma unroll 1
            for (int s = 0; s < 2 * NBOX; ++s) {
              const int which = s / NBOX, box = s % NBOX, slot = s & 1;
              if (s == 0 || s >= 2) {  // the slot's last reader (the dQ reduction, or stage s-2) is done
                if (threadIdx.x == 256) {
                  if (s == 0)
                    bulk_wait_read_all();
                  else
                    bulk_wait_read_all_but_newest();
                  mbar_arrive(&bars->kvst_free);
                }
                if (!mbar_wait(&bars->kvst_free, kvst_free_ph, ab)) goto done;
                kvst_free_ph ^= 1;
              }
              const uint32_t tAcc = tmem + lane_addr + (which == 0 ? C::COL_DV : C::COL_DK);
              const float mul = which == 0 ? 1.0f : p.scale;
#pragma unroll 1
              for (int c = 64 * box; c < 64 * box + 64; c += 32) {
                uint32_t ov[32];
                tmem_ld32(tAcc + c, ov);
                tmem_wait_ld();
                reg_fence<32>(ov);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  pk[e] = pack_bf16(__uint_as_float(ov[2 * e]) * mul, __uint_as_float(ov[2 * e + 1]) * mul);
                // row r of the slot's 64-column box, 16-byte pieces (c%64)/8 .. +3, 128-byte swizzle
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const uint32_t addr = stage32 + slot * 16384 + r * 128 + ((((c % 64) / 8 + e) ^ (r & 7)) << 4);
                  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * e]),
                               "r"(pk[4 * e + 1]), "r"(pk[4 * e + 2]), "r"(pk[4 * e + 3])
                               : "memory");
                }
              }
              if (s == 2 * NBOX - 1) {  // dV and dK are out of TMEM: the next unit's MMAs may start
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->dkv_empty);
              }
              fence_proxy_async_smem();
              mbar_arrive(&bars->kvst_full);
              if (!mbar_wait(&bars->kvst_full, kvst_full_ph, ab)) goto done;
              kvst_full_ph ^= 1;
              if (threadIdx.x == 256) {
                tma_store_2d(which == 0 ? &tm_dv : &tm_dk, smem + C::OFF_STG + slot * 16384, u.h * D + 64 * box,
                             u.kv0 + BK * u.n);
                bulk_commit_group();
              }
            }
            // hand the buffer back to the dQ reduction
            if (threadIdx.x == 256) {
              bulk_wait_read_all();
              mbar_arrive(&bars->kvst_free);
            }
            if (!mbar_wait(&bars->kvst_free, kvst_free_ph, ab)) goto done;
            kvst_free_ph ^= 1;
          } else {
  #pragma unroll 1
            for (int which = 0; which < 2; ++which) {
              if (full_blk) {  // the buffer holds nothing TMA still reads
                if (threadIdx.x == 256) {
                  bulk_wait_read_all();
                  mbar_arrive(&bars->kvst_free);
                }
                if (!mbar_wait(&bars->kvst_free, kvst_free_ph, ab)) goto done;
                kvst_free_ph ^= 1;
              }
              const uint32_t tAcc = tmem + lane_addr + (which == 0 ? C::COL_DV : C::COL_DK);
              const float mul = which == 0 ? 1.0f : p.scale;
              __nv_bfloat16* dst = (which == 0 ? p.dv : p.dk) + row;
  #pragma unroll 1
              for (int c = 0; c < D; c += 32) {
                uint32_t ov[32];
                tmem_ld32(tAcc + c, ov);
                tmem_wait_ld();
                reg_fence<32>(ov);
                uint32_t pk[16];
  #pragma unroll
                for (int e = 0; e < 16; ++e)
                  pk[e] = pack_bf16(__uint_as_float(ov[2 * e]) * mul, __uint_as_float(ov[2 * e + 1]) * mul);
                if (full_blk) {
                  // row r of 64-column box c/64, 16-byte pieces (c%64)/8 .. +3, 128-byte swizzle
  #pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const uint32_t addr =
                        stage32 + (c / 64) * 16384 + r * 128 + ((((c % 64) / 8 + e) ^ (r & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * e]),
                                 "r"(pk[4 * e + 1]), "r"(pk[4 * e + 2]), "r"(pk[4 * e + 3])
                                 : "memory");
                  }
                } else if (key_ok) {
  #pragma unroll
                  for (int e = 0; e < 4; ++e)
                    st_global_v4(dst + c + 8 * e, pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                }
              }
              if (which == 1) {  // dV and dK are out of TMEM: the next unit's MMAs may start
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->dkv_empty);
              }
              if (full_blk) {
                fence_proxy_async_smem();
                mbar_arrive(&bars->kvst_full);
                if (!mbar_wait(&bars->kvst_full, kvst_full_ph, ab)) goto done;
                kvst_full_ph ^= 1;
                if (threadIdx.x == 256) {
  #pragma unroll
                  for (int b2 = 0; b2 < D / 64; ++b2)
                    tma_store_2d(which == 0 ? &tm_dv : &tm_dk, smem + C::OFF_STG + b2 * 16384, u.h * D + 64 * b2,
                                 u.kv0 + BK * u.n);
                  bulk_commit_group();
                }
              }
            }
            if (full_blk) {  // hand the buffer back to the dQ reduction
              if (threadIdx.x == 256) {
                bulk_wait_read_all();
                mbar_arrive(&bars->kvst_free);
              }
              if (!mbar_wait(&bars->kvst_free, kvst_free_ph, ab)) goto done;
              kvst_free_ph ^= 1;
            }
          }
        }
        if (!mbar_wait(&bars->dq_full, ph, ab)) goto done;
        ph ^= 1;
        tc_fence_after();
        // the whole row into registers first, then TMEM goes back to the MMA warp
        uint32_t v[D];
#pragma unroll
        for (int c = 0; c < D; c += 32) tmem_ld32(tQ + c, v + c);
        tmem_wait_ld();
        reg_fence<D>(v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->dq_empty);
        // Stage the rows in shared memory and reduce-add them into the fp32
        // accumulator with TMA (aixai.ru summary, "dQ epilogue": staged
        // writeback): one 32-column swizzled box per round, alternating between
        // two 16 KB slots, so the rows of round g are written while TMA still
        // reads round g-1; one box is read at a time (more in flight slowed the
        // TMA loads that share the engine).  Rows past the end of the query set
        // are exactly zero (their P is zero), so adding them is harmless, and
        // TMA clips rows past the end of the tensor.
        uint8_t* stage = smem + C::OFF_STG;
        const uint32_t stage_u32 = smem_u32(stage);
        const int y = u.q_base + BQ * i;
        uint32_t g = q_it * (D / 32);  // rounds so far (the same count in every drain thread)
#pragma unroll
        for (int rnd = 0; rnd < D / 32; ++rnd, ++g) {
          const uint32_t slot = g & 1;
          if (g >= 2) {  // slot last read by the TMA of round g-2
            if (threadIdx.x == 256) {
              bulk_wait_read_all_but_newest();
              mbar_arrive(&bars->stg_free[slot]);
            }
            if (!mbar_wait(&bars->stg_free[slot], ((g >> 1) - 1) & 1, ab)) goto done;
          }
          const uint32_t row = stage_u32 + slot * 16384 + r * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int c = 32 * rnd + 4 * j;
            const uint32_t addr = row + ((j ^ (r & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[c]), "r"(v[c + 1]),
                         "r"(v[c + 2]), "r"(v[c + 3])
                         : "memory");
          }
          fence_proxy_async_smem();
          mbar_arrive(&bars->stg_full[slot]);
          if (!mbar_wait(&bars->stg_full[slot], (g >> 1) & 1, ab)) goto done;
          if (threadIdx.x == 256) {
            bulk_wait_read_all();  // one box being read at a time
            tma_reduce_add_2d(&tm_dq, stage + slot * 16384, (u.h * p.G + hg) * D + 32 * rnd, y);
            bulk_commit_group();
          }
        }
      }
    }
    if (threadIdx.x == 256) bulk_wait_all();
  } else {
    setmaxnreg_dec<kRegIssue>();
    if (warp == 12) {
      if (lane == 0) {
        // ------------------------------------------------------ MMA issuer
        const uint32_t id_s = idesc_bf16(128, 128, 0, 0);   // S^T, dP^T
        const uint32_t id_kv = idesc_bf16(128, D, 0, 1);    // dV, dK: B (dO, Q) MN-major
        const uint32_t id_q = idesc_bf16(128, D, 1, 1);     // dQ: A (dS) and B (K) MN-major
        const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
        const uint32_t sDS = smem_u32(smem + C::OFF_DS);
        uint32_t kv_ph = 0, ph = 0, dq_ph = 0, dkv_ph = 0, q_it = 0;
        // S^T = K Q^T of tile t into its region; false if the CTA aborts
        auto issue_s = [&](uint32_t t) -> bool {
          const uint32_t st_t = t & 1;
          if (!mbar_wait(&bars->q_full[st_t], (t >> 1) & 1, ab)) return false;
          tc_fence_after();
          const uint32_t sQt = smem_u32(smem + C::OFF_Q + st_t * C::TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
            mma_ss(tmem + region_s(t), sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQt + off, 16, 1024), id_s,
                   kk > 0);
          }
          mma_commit(&bars->s_full);
          return true;
        };
        for (uint32_t it = 0;; ++it) {
          const int ui = sched_pop(bars, it, ab, false);
          if (ui == -2) goto mma_done;
          if (ui < 0) break;
          const Unit u = decode<MASK>(p, ui);
          if (!mbar_wait(&bars->kv_full, kv_ph, ab)) goto mma_done;
          kv_ph ^= 1;
          if (!issue_s(q_it)) goto mma_done;  // the unit's first tile
          for (int hg = 0; hg < p.G; ++hg)
          for (int i = u.i0; i < u.i1; ++i, ++q_it) {
            const bool first = hg == 0 && i == u.i0;          // the unit's first tile
            const bool last = hg + 1 == p.G && i + 1 == u.i1;  // and its last
            const uint32_t st = q_it & 1;
            const uint32_t sQ = smem_u32(smem + C::OFF_Q + st * C::TILE);
            const uint32_t sDO = smem_u32(smem + C::OFF_DO);
            // S^T and dP^T swap TMEM regions every tile: S^T goes where the
            // previous dP^T was (already consumed), dP^T where the previous S^T
            // was, which holds the previous tile's dQ until the drain has read it.
            const uint32_t rs = region_s(q_it), rd = 128 - rs;
            // dP^T = V dO^T, once the previous dQ has left TMEM
            if (!first || it > 0) {
              if (!mbar_wait(&bars->dq_empty, dq_ph, ab)) goto mma_done;
              dq_ph ^= 1;
            }
            if (!mbar_wait(&bars->do_full, q_it & 1, ab)) goto mma_done;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
              mma_ss(tmem + rd, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sDO + off, 16, 1024), id_s, kk > 0);
            }
            mma_commit(&bars->dp_full);
            // dV += P^T dO  (A from TMEM)
            if (first) {
              if (!mbar_wait(&bars->dkv_empty, dkv_ph ^ 1, ab)) goto mma_done;
              dkv_ph ^= 1;
            }
            if (!mbar_wait(&bars->p_full, ph, ab)) goto mma_done;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t pcol = (kk < 4) ? 8 * kk : 64 + 8 * (kk - 4);
              mma_ts(tmem + C::COL_DV, tmem + rs + pcol, sdesc_sw128(sDO + kk * 2048, C::CHUNK, 1024), id_kv,
                     (!first || kk > 0) ? 1u : 0u);
            }
            mma_commit(&bars->do_empty);  // dV was dO's last reader: the next dO may load
            if (!mbar_wait(&bars->ds_full, ph, ab)) goto mma_done;
            ph ^= 1;
            tc_fence_after();
            // dQ = dS K first (the drain can start), then the next tile's S^T into
            // this tile's dP^T region (read by the dS phase that just finished),
            // then dK += dS^T Q: the next tile's P phase overlaps dK.
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tmem + rs, sdesc_sw128(sDS + kk * 2048, C::CHUNK, 1024), sdesc_sw128(sK + kk * 2048, C::CHUNK, 1024),
                     id_q, kk > 0);
            mma_commit(&bars->dq_full);
            if (!last && !issue_s(q_it + 1)) goto mma_done;
            if (last) mma_commit(&bars->kv_empty);  // K and V are done: the next unit's may load
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
              mma_ss(tmem + C::COL_DK, sdesc_sw128(sDS + off, 16, 1024), sdesc_sw128(sQ + kk * 2048, C::CHUNK, 1024),
                     id_kv, (!first || kk > 0) ? 1u : 0u);
            }
            mma_commit(&bars->ds_empty);
            mma_commit(&bars->q_empty[st]);
          }
          mma_commit(&bars->dkv_full);
        }
      mma_done:
        mma_commit(&bars->drain);
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&bars->drain, 0) && global_timer_ns() - t0 < kWaitTimeoutNs) {
        }
      }
    } else if (warp == 13) {
      // ------------------------------------------------------ loader and scheduler (whole warp)
      // Static plan: this CTA's slice of the list.  Cluster Launch Control: the
      // CTA starts with its own index and, while loading a unit, asks the
      // hardware for a CTA that has not launched yet and takes over its unit
      // (aixai.ru summary, "Tile balancing and Cluster Launch Control").
      uint32_t kv_ph = 0, q_it = 0;
      bool ok = true;
      int cur = p.use_clc ? static_cast<int>(blockIdx.x) : (u_begin < u_end ? u_begin : -1);
      for (uint32_t it = 0; ok; ++it) {
        const int slot = it & 3;
        if (!mbar_wait(&bars->sched_empty[slot], ((it >> 2) & 1) ^ 1, ab)) break;
        if (lane == 0) {
          bars->sched_unit[slot] = cur;
          mbar_arrive(&bars->sched_full[slot]);
          if (cur >= 0 && p.use_clc) {
            mbar_expect_tx(&bars->clc_bar, 16);
            clc_try_cancel(&bars->clc_resp, &bars->clc_bar);
          }
        }
        if (cur < 0) break;
        const Unit u = decode<MASK>(p, cur);
        if (!mbar_wait(&bars->kv_empty, kv_ph ^ 1, ab)) break;
        kv_ph ^= 1;
        if (lane == 0) {
          mbar_expect_tx(&bars->kv_full, 2 * C::TILE);
#pragma unroll
          // K and V are read by this unit only: first out of L2; the query tiles
          // and dO are read again by the sequence's other key blocks: last out
          for (int c = 0; c < D / 64; ++c) {
            tma_load_2d_hint(&tm_k, &bars->kv_full, smem + C::OFF_K + c * C::CHUNK, u.h * D + c * 64, u.kv0 + BK * u.n,
                             l2_policy_evict_first());
            tma_load_2d_hint(&tm_v, &bars->kv_full, smem + C::OFF_V + c * C::CHUNK, u.h * D + c * 64, u.kv0 + BK * u.n,
                             l2_policy_evict_first());
          }
        }
        for (int hg = 0; hg < p.G && ok; ++hg)
        for (int i = u.i0; i < u.i1; ++i, ++q_it) {
          const int hq = u.h * p.G + hg;  // query head
          const uint32_t st = q_it & 1;
          if (!mbar_wait(&bars->q_empty[st], ((q_it >> 1) & 1) ^ 1, ab)) {
            ok = false;
            break;
          }
          // L and Di of the tile's 128 query rows (rows past the end: L = +inf so P = 0)
          const size_t lbase = static_cast<size_t>(hq) * p.o_rows + u.o_base + BQ * i;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = 4 * lane + e;
            const bool v = BQ * i + r < u.rows;
            s_lse[st * 128 + r] = v ? p.lse2[lbase + r] : INFINITY;
            s_di[st * 128 + r] = v ? p.di[lbase + r] : 0.f;
          }
          uint8_t* sQ = smem + C::OFF_Q + st * C::TILE;
          if (lane == 0) {
            mbar_expect_tx(&bars->q_full[st], C::TILE);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_load_2d_hint(&tm_q, &bars->q_full[st], sQ + c * C::CHUNK, hq * D + c * 64, u.q_base + BQ * i,
                               l2_policy_evict_last());
          } else {
            mbar_arrive(&bars->q_full[st]);
          }
          // dO: a single buffer, free once the previous tile's dV has read it
          if (!mbar_wait(&bars->do_empty, (q_it & 1) ^ 1, ab)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_expect_tx(&bars->do_full, C::TILE);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_load_2d_hint(&tm_do, &bars->do_full, smem + C::OFF_DO + c * C::CHUNK, hq * D + c * 64,
                               u.o_base + BQ * i, l2_policy_evict_last());
          }
        }
        if (!ok) break;
        if (p.use_clc) {
          // lane 0 alone reads the response (before it issues the next request
          // into the same buffer) and hands it to the warp
          int got = 1, nxt = -1;
          if (lane == 0) {
            got = mbar_wait(&bars->clc_bar, it & 1, ab) ? 1 : 0;
            if (got) nxt = clc_cancelled_x(&bars->clc_resp);
          }
          if (!__shfl_sync(0xffffffffu, got, 0)) break;
          cur = __shfl_sync(0xffffffffu, nxt, 0);
          if (cur >= p.n_units) cur = -1;
        } else {
          cur = cur + 1 < u_end ? cur + 1 : -1;
        }
      }
      if (*ab.flag) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 100000000ull) {
        }
      }
    }
  }
done:
  __syncwarp();
  __syncthreads();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Di[h, r] = sum_d dO[r,h,d] O[r,h,d];  lse2[h, r] = L[h, r] log2(e).
// 16 threads per (row, head) for D = 128 (8 per head for D = 64), 8 bf16 each.
// Di and L * log2(e) for every (head, row) pair, and a zero fill of the fp32
// dQ accumulator that the main kernel reduce-adds into.  Pairs are numbered
// head-major (p = h * rows + r, the layout of L and Di), so consecutive pairs are
// consecutive rows of one head and the per-pair results are written coalesced;
// each pair's O and dO rows (D bf16 each) are read by D/8 lanes with 16-byte
// loads, several pairs per thread in flight.
template <int D>
__global__ void prep_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                            const float* __restrict__ lse, float* __restrict__ di, float* __restrict__ lse2,
                            int rows, int H, float4* __restrict__ acc, long acc4) {
  constexpr int TPP = D / 8;     // lanes per pair
  constexpr int PPW = 32 / TPP;  // pairs per warp per round
  constexpr int U = 2;           // rounds whose loads are in flight together
  const int lane = threadIdx.x & 31, part = lane % TPP;
  const long warp = (static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long n_warps = (static_cast<long>(gridDim.x) * blockDim.x) >> 5;
  const long n_pairs = static_cast<long>(rows) * H;
  for (long base = warp * PPW * U; base < n_pairs; base += n_warps * PPW * U) {
    uint4 a[U], b[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long pr = base + u * PPW + lane / TPP;
      if (pr < n_pairs) {
        const long h = pr / rows, r = pr - h * rows;
        const size_t at = (static_cast<size_t>(r) * H + h) * D + part * 8;
        a[u] = ld_stream_v4(o + at);
        b[u] = ld_stream_v4(dout + at);
      } else {
        a[u] = make_uint4(0, 0, 0, 0);
        b[u] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[u]);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b[u]);
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __bfloat1622float2(a2[e]);
        const float2 fb = __bfloat1622float2(b2[e]);
        s = fmaf(fa.x, fb.x, s);
        s = fmaf(fa.y, fb.y, s);
      }
#pragma unroll
      for (int off = TPP / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      const long pr = base + u * PPW + lane / TPP;
      if (part == 0 && pr < n_pairs) {
        di[pr] = s;
        lse2[pr] = lse[pr] * kLog2e;
      }
    }
  }
  for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < acc4;
       i += static_cast<long>(gridDim.x) * blockDim.x)
    st_global_v4(acc + i, 0u, 0u, 0u, 0u);
}

__global__ void dq_convert_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq, long n4, float scale) {
  for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += static_cast<long>(gridDim.x) * blockDim.x) {
    const uint4 raw = ld_stream_v4(reinterpret_cast<const float4*>(acc) + i);
    const float4 v = make_float4(__uint_as_float(raw.x), __uint_as_float(raw.y), __uint_as_float(raw.z),
                                 __uint_as_float(raw.w));
    st_global_v2(reinterpret_cast<uint2*>(dq) + i, pack_bf16(v.x * scale, v.y * scale), pack_bf16(v.z * scale, v.w * scale));
  }
}

template <int D, int MASK, bool FINE = false>
int launch_main(const BwdArgs& a) {
  using C = Cfg<D>;
  CUtensorMap tq, tk, tv, tdo;
  int st = make_map_2d(&tq, a.q, static_cast<uint64_t>(a.H) * D, a.q_rows, 64, BQ);
  if (st == JFA_OK) st = make_map_2d(&tk, a.k, static_cast<uint64_t>(a.Hkv) * D, a.kv_rows, 64, BK);
  if (st == JFA_OK) st = make_map_2d(&tv, a.v, static_cast<uint64_t>(a.Hkv) * D, a.kv_rows, 64, BK);
  if (st == JFA_OK) st = make_map_2d(&tdo, a.dout, static_cast<uint64_t>(a.H) * D, a.o_rows, 64, BQ);
  CUtensorMap tdq;  // fp32 dQ accumulator, 32-column boxes for the staged reduce-add
  if (st == JFA_OK) st = make_map_2d_f32(&tdq, a.dq_acc, static_cast<uint64_t>(a.H) * D, a.q_rows, 32, BQ);
  CUtensorMap tdk, tdv;  // dK, dV outputs: 64-column boxes of one 128-key block
  if (st == JFA_OK) st = make_map_2d(&tdk, a.dk, static_cast<uint64_t>(a.Hkv) * D, a.kv_rows, 64, BK);
  if (st == JFA_OK) st = make_map_2d(&tdv, a.dv, static_cast<uint64_t>(a.Hkv) * D, a.kv_rows, 64, BK);
  if (st != JFA_OK) return st;
  auto kern = bwd_kernel<D, MASK, FINE>;
  static PerDeviceOnce setup;  // per instantiation
  st = setup.run([&]() -> int {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return JFA_ERR_CUDA;
    if (fa.numRegs * kThreads < kRegTotal) return JFA_ERR_UNSUPPORTED;  // the split could never be granted
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC) != cudaSuccess)
      return JFA_ERR_CUDA;
    return JFA_OK;
  });
  if (st != JFA_OK) return st;
  Params p;
  p.units = reinterpret_cast<const int4*>(a.units);
  p.cta_start = a.cta_start;
  p.offsets = a.offsets_dev;
  p.lse2 = a.lse2;
  p.di = a.di;
  p.dq_acc = a.dq_acc;
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.err = a.err;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.G = a.H / a.Hkv;
  p.nq = a.nq;
  p.o_rows = a.o_rows;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.use_clc = a.use_clc;
  p.n_units = a.n_units;
  p.win_left = a.win_left;
  p.win_right = a.win_right;
  ProfileScope prof(kKindBwdMain, a.stream);
  kern<<<a.use_clc ? a.n_units : a.n_cta, kThreads, C::SMEM_ALLOC, a.stream>>>(tq, tk, tv, tdo, tdq, tdk, tdv, p);
  return cudaGetLastError() == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

}  // namespace bwd

int launch_bwd_prep(const BwdArgs& a, int num_sms) {
  const long pairs = static_cast<long>(a.o_rows) * a.H;
  const long acc4 = static_cast<long>(a.q_rows) * a.H * a.D / 4;
  if (pairs == 0 && acc4 == 0) return JFA_OK;
  const int block = 256;
  // enough warps for every pair to be visited once where that fits, capped at
  // one wave (48 registers: 5 blocks of 256 per SM); larger problems loop
  const long per_block = (block / 32) * (32 / (a.D / 8)) * 2;
  long grid = std::max((pairs + per_block - 1) / per_block, (acc4 + block - 1) / block);
  grid = std::min<long>(std::max<long>(grid, 1), 5L * num_sms);
  ProfileScope prof(kKindBwdPrep, a.stream);
  float4* acc = reinterpret_cast<float4*>(a.dq_acc);
  if (a.D == 128)
    bwd::prep_kernel<128><<<static_cast<int>(grid), block, 0, a.stream>>>(
        static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dout), a.lse, a.di, a.lse2,
        a.o_rows, a.H, acc, acc4);
  else
    bwd::prep_kernel<64><<<static_cast<int>(grid), block, 0, a.stream>>>(
        static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dout), a.lse, a.di, a.lse2,
        a.o_rows, a.H, acc, acc4);
  return cudaGetLastError() == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

int launch_bwd_main(const BwdArgs& a) {
  if (a.D == 128) {
    if (a.mask == kMaskWindow) return bwd::launch_main<128, kMaskWindow>(a);
    if (a.mask == kMaskCausal) return bwd::launch_main<128, kMaskCausal>(a);
    return a.nq > 0 ? bwd::launch_main<128, kMaskNone, true>(a) : bwd::launch_main<128, kMaskNone>(a);
  }
  if (a.mask == kMaskWindow) return bwd::launch_main<64, kMaskWindow>(a);
  if (a.mask == kMaskCausal) return bwd::launch_main<64, kMaskCausal>(a);
  return a.nq > 0 ? bwd::launch_main<64, kMaskNone, true>(a) : bwd::launch_main<64, kMaskNone>(a);
}

int launch_dq_convert(const BwdArgs& a, int num_sms) {
  const long n4 = static_cast<long>(a.q_rows) * a.H * a.D / 4;
  if (n4 == 0) return JFA_OK;
  long grid = (n4 + 255) / 256;
  if (grid > 8L * num_sms) grid = 8L * num_sms;
  ProfileScope prof(kKindDqConvert, a.stream);
  bwd::dq_convert_kernel<<<static_cast<int>(grid), 256, 0, a.stream>>>(a.dq_acc, static_cast<__nv_bfloat16*>(a.dq),
                                                                       n4, a.scale);
  return cudaGetLastError() == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

}  // namespace jfa
