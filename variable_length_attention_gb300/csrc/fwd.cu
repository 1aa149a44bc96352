// fwd.cu -- jagged flash-attention forward for sm_103a.
//
// What it computes: for every packed sequence and head, O = softmax(scale Q K^T) V
// and the natural-log log-sum-exp of each score row, with the online-softmax
// recurrence of the standard flash-attention loop ("TLX Block Attention",
// section 2.1, Listing 1): a running row maximum m and sum l, a correction
// factor when m grows, O = acc / l at the end, L = m + log(l) stored for the
// backward pass.
//
// How (one persistent CTA per SM, warp-specialised; the role split follows the
// aixai.ru summary, "Framework", and the commentary page, "architecture"):
//   warps 0-3   softmax of query tile 0 (one thread per row = one TMEM lane)
//   warps 4-7   softmax of query tile 1
//   warps 8-11  epilogue: O / l -> bf16 -> global, log-sum-exp
//   warp 12     tcgen05 MMA issuer (one thread)
//   warp 13     TMA loader (one thread): Q tiles, then a K/V ring in shared memory
// A work unit is 256 query rows (two 128-row tiles) of one (sequence, head); both
// tiles share every K/V block the loader brings in.  The MMA warp interleaves
// the two tiles so the tensor core computes one tile's S = Q K^T while the
// other tile's softmax runs:  S0 S1 | PV0 S0' PV1 S1' | PV0 S0'' ...
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [384,384+D);
// P (bf16, two per column) overwrites the first 64 columns of its S.
// The running maximum is only moved (and O rescaled) when it grows by more than
// 2^8; otherwise the stale maximum is kept, which is exact because numerator and
// denominator share it.
// Keys past the end of a sequence and, for causal attention or a sliding
// window, keys outside the row's window are masked in separate, peeled
// iterations so the main loop has no mask (aixai.ru summary, "Loop peeling
// against register spills").  With a window each query tile visits only the
// K/V blocks its rows can see: tile 1 may start a block later than tile 0 and
// tile 0 may stop a block earlier.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "host.h"
#include "profile.h"
#include "ptx.cuh"

namespace jfa {
namespace fwd {

constexpr int BM = 128;  // rows per query tile
constexpr int BN = 128;  // keys per K/V block
constexpr int kThreads = 512;
// Registers per thread after the warpgroups' setmaxnreg: two softmax
// warpgroups, the epilogue warpgroup, the MMA/loader warpgroup.  Their sum must
// not exceed what the CTA is launched with (128 per thread at 512 threads), or
// setmaxnreg.inc would wait forever; the launcher checks the compiled count.
// The sliding-window softmax keeps its window bounds as well and takes 8 more.
template <int MASK>
struct RegSplit {
  static constexpr int kSoftmax = MASK == kMaskWindow ? 184 : 176;
  static constexpr int kEpilogue = MASK == kMaskWindow ? 56 : 64;
  static constexpr int kIssue = MASK == kMaskWindow ? 88 : 96;
  static constexpr int kTotal = 2 * 128 * kSoftmax + 128 * kEpilogue + 128 * kIssue;
  static_assert(kTotal <= kThreads * 128, "register split exceeds the launch allocation");
};
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct Cfg {
  static constexpr int NCHUNK = D / 64;                  // 128-byte swizzle atoms across head_dim
  static constexpr int TILE_BYTES = BM * D * 2;          // one Q tile or one K/V block
  static constexpr int CHUNK_BYTES = BM * 128;           // one 64-column box
  static constexpr int NSTAGE = D == 128 ? 4 : 6;        // K/V ring depth
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = 2 * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_KV + NSTAGE * TILE_BYTES;
  static constexpr int OFF_STG = OFF_BAR + 4096;         // after barriers, stats, TMEM address:
  static constexpr int SMEM_BYTES = OFF_STG + BM * 128;  // O staging, one 64-column bf16 box
  static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;   // slack for 1024-byte alignment
};

struct Params {
  __nv_bfloat16* o;
  float* lse;
  const int32_t* offsets;
  const int4* units;
  const int32_t* cta_start;  // static plan: CTA c takes units [cta_start[c], cta_start[c+1])
  int* err;
  int H, Hkv, nq, o_rows;
  int n_units;
  int use_clc;               // 1: one CTA per unit in cost order, idle CTAs claim pending ones
  int win_left, win_right;   // sliding window (kMaskWindow): keys [row - left, row + right], -1 = open
  const int32_t* topk_sel;   // block-sparse (kMaskTopK): chosen key blocks [query blocks, topk]
  const int32_t* topk_qb;    // query blocks before each sequence [batch+1]
  int topk;
  float scale_log2;
};

struct Unit {
  int b, h, g, m;
  int kv0, L;       // first K/V row, K/V length
  int rows;         // query rows of the sequence (self) or of the shared Q (broadcast)
  int q_row0;       // first query row of the unit in q
  int o_row0;       // first output row of the unit in o
  int j0, n_kv;     // K/V blocks loaded: j0 .. j0 + n_kv - 1
  int je0;          // tile 0 visits blocks [j0, je0) (causal: it skips the unit's last block when
                    // that block lies wholly in its masked future)
  int jb1, je1;     // tile 1 visits blocks [jb1, je1)
  int pb0, pe0;     // tile 0: blocks in [pb0, pe0) need no mask
  int pb1, pe1;     // tile 1: the same
  int nt;           // query tiles of the unit: 1 when the second tile lies wholly past the last row
  const int32_t* sel;  // block-sparse: the unit's chosen key blocks (block j of the loop is sel[j])
  int tail_hi;         // block-sparse: valid keys of the sequence's last block
};

// Block range [*jb, *je) a query tile whose rows are [r, last] sees under a
// window, and the range [*pb, *pe) of those blocks that every row sees whole.
__device__ __forceinline__ void window_blocks(int r, int last, int L, int left, int right, int* jb, int* je,
                                              int* pb, int* pe) {
  const int lo = left < 0 ? 0 : max(0, r - left);
  const int hi = right < 0 ? L : min(L, last + right + 1);
  *jb = lo / BN;
  *je = (hi + BN - 1) / BN;
  *pb = (left < 0 || last - left <= 0) ? 0 : (last - left + BN - 1) / BN;
  *pe = right < 0 ? L / BN : min(L / BN, (r + right + 1) / BN);
}

template <int MASK>
__device__ __forceinline__ Unit decode(const Params& p, int idx) {
  const int4 e = p.units[idx];
  Unit u;
  u.b = e.x;
  u.h = e.y;
  u.m = e.z;
  u.g = u.h / (p.H / p.Hkv);
  u.kv0 = p.offsets[u.b];
  u.L = e.w;  // the sequence length (the host wrote it into the entry)
  if (p.nq > 0) {
    u.rows = p.nq;
    u.q_row0 = 2 * BM * u.m;
    u.o_row0 = u.b * p.nq + 2 * BM * u.m;
  } else {
    u.rows = u.L;
    u.q_row0 = u.kv0 + 2 * BM * u.m;
    u.o_row0 = u.q_row0;
  }
  u.nt = 2 * BM * u.m + BM < u.rows ? 2 : 1;
  u.j0 = 0;
  u.jb1 = 0;
  u.pb0 = u.pb1 = 0;
  if (MASK == kMaskCausal) {
    const int last = min(2 * BM * (u.m + 1), u.rows);
    u.n_kv = (min(last, u.L) + BN - 1) / BN;
    u.pe0 = u.pe1 = min(u.L / BN, 2 * u.m);
    u.je0 = min(u.n_kv, 2 * u.m + 1);
    u.je1 = u.n_kv;
  } else if (MASK == kMaskWindow) {  // self-attention only: rows = L
    const int r0 = 2 * BM * u.m;
    int je1 = 0;
    window_blocks(r0, min(r0 + BM, u.L) - 1, u.L, p.win_left, p.win_right, &u.j0, &u.je0, &u.pb0, &u.pe0);
    if (u.nt == 2)
      window_blocks(r0 + BM, min(r0 + 2 * BM, u.L) - 1, u.L, p.win_left, p.win_right, &u.jb1, &je1, &u.pb1,
                    &u.pe1);
    u.je1 = je1;
    u.n_kv = max(u.je0, je1) - u.j0;
  } else if (MASK == kMaskTopK) {  // the chosen blocks, in ascending order
    const int nblk = (u.L + BN - 1) / BN;
    const int q0 = p.topk_qb[u.b];
    const int row = p.H * q0 + u.h * (p.topk_qb[u.b + 1] - q0) + u.m;
    u.sel = p.topk_sel + static_cast<size_t>(row) * p.topk;
    u.n_kv = min(p.topk, nblk);
    u.je0 = u.je1 = u.n_kv;
    // only the sequence's last block can be short; chosen, it is the last in the list
    const bool tail = (u.L % BN) != 0 && u.sel[u.n_kv - 1] == nblk - 1;
    u.pe0 = u.pe1 = tail ? u.n_kv - 1 : u.n_kv;
    u.tail_hi = u.L - (nblk - 1) * BN;
  } else {
    u.n_kv = (u.L + BN - 1) / BN;
    u.pe0 = u.pe1 = u.L / BN;
    u.je0 = u.je1 = u.n_kv;
  }
  return u;
}

struct Bars {
  uint64_t q_full[2];
  uint64_t q_empty;
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_full[2];
  uint64_t o_empty[2];
  uint64_t st_full[2];
  uint64_t st_empty[2];
  uint64_t drain;
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  // unit schedule: the loader publishes each unit index (or -1 at the end) to
  // every role through this ring
  uint64_t sched_full[4], sched_empty[4], clc_bar;
  int4 clc_resp;
  int sched_unit[4];
  float stat_m[2][BM];
  float stat_l[2][BM];
  uint64_t ostg_full, ostg_free;  // O staging box: rows written by the epilogue / read out by TMA
  uint32_t tmem_base;
  int abort_flag;
};

constexpr int kSchedConsumers = 13;  // MMA thread + 8 softmax warps + 4 epilogue warps


template <int D, int MASK>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, const Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sKV = smem + C::OFF_KV;
  Bars* bars = reinterpret_cast<Bars*>(smem + C::OFF_BAR);
  static_assert(sizeof(Bars) <= 4096, "barrier block too large");

  const int warp = warp_id();
  const int lane = lane_id();
  const int u_begin = p.use_clc ? 0 : p.cta_start[blockIdx.x];
  const int u_end = p.use_clc ? 0 : p.cta_start[blockIdx.x + 1];

  if (threadIdx.x == 0) {
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bars->sched_full[s], 1);
      mbar_init(&bars->sched_empty[s], kSchedConsumers);
    }
    mbar_init(&bars->clc_bar, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->q_full[t], 1);
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 4);
      mbar_init(&bars->o_full[t], 1);
      mbar_init(&bars->o_empty[t], BM);
      mbar_init(&bars->st_full[t], BM);
      mbar_init(&bars->st_empty[t], BM);
    }
    mbar_init(&bars->q_empty, 1);
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->ostg_full, BM);
    mbar_init(&bars->ostg_free, 1);
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
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
    // ------------------------------------------------------------ softmax
    setmaxnreg_inc<RegSplit<MASK>::kSoftmax>();
    const int t = warp >> 2;                 // query tile of this warpgroup
    const int row = threadIdx.x & 127;       // TMEM lane == row of the tile
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_addr + t * BN;
    const uint32_t tO = tmem + lane_addr + 256 + t * 128;
    const float sl2 = p.scale_log2;
    uint32_t s_phase = 0, st_phase = 0;
    for (uint32_t it = 0;; ++it) {
      const int ui = sched_pop(bars, it, ab, true);
      if (ui == -2) goto done;
      if (ui < 0) break;
      const Unit u = decode<MASK>(p, ui);
      if (t >= u.nt) continue;                     // a single-tile unit: nothing for tile 1
      const int qi = 2 * BM * u.m + BM * t + row;  // query index inside the sequence / shared Q
      float m_run = -INFINITY, l_run = 0.f;
      // blocks [jb, je) of the tile; those in [pb, pe) need no mask (without a
      // window every tile starts at block 0 and only trailing blocks are masked)
      constexpr bool kRanged = MASK == kMaskWindow || MASK == kMaskTopK;
      const int jb = kRanged ? (t == 0 ? u.j0 : u.jb1) : 0, je = t == 0 ? u.je0 : u.je1;
      const int pb = MASK == kMaskWindow ? (t == 0 ? u.pb0 : u.pb1) : 0, pe = t == 0 ? u.pe0 : u.pe1;
      for (int j = jb; j < je; ++j) {
        if (!mbar_wait(&bars->s_full[t], s_phase, ab)) goto done;
        s_phase ^= 1;
        tc_fence_after();
        uint32_t sr[BN];
        tmem_ld32(tS + 0, sr + 0);
        tmem_ld32(tS + 32, sr + 32);
        tmem_ld32(tS + 64, sr + 64);
        tmem_ld32(tS + 96, sr + 96);
        tmem_wait_ld();
        reg_fence<BN>(sr);
        float s[BN];
#pragma unroll
        for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(sr[c]);
        if ((MASK == kMaskWindow && j < pb) || j >= pe) {  // peeled tail / diagonal / window-edge iterations
          // visible key columns of this block: [lo, hi)
          const int wr = MASK == kMaskCausal ? 0 : (MASK == kMaskWindow ? p.win_right : -1);
          const int hi = MASK == kMaskTopK ? u.tail_hi : (wr < 0 ? u.L : min(u.L, qi + wr + 1)) - j * BN;
          if (MASK == kMaskWindow) {
            const int lo = p.win_left < 0 ? -BN : qi - p.win_left - j * BN;
#pragma unroll
            for (int c = 0; c < BN; ++c)
              if (c >= hi || c < lo) s[c] = -INFINITY;
          } else {
#pragma unroll
            for (int c = 0; c < BN; ++c)
              if (c >= hi) s[c] = -INFINITY;
          }
        }
        // row maximum: 4 independent partial maxima, two new values per step
        float pm[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) pm[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
        for (int c = 8; c < BN; c += 8)
#pragma unroll
          for (int i = 0; i < 4; ++i) pm[i] = fmax3(pm[i], s[c + 2 * i], s[c + 2 * i + 1]);
        const float mx = fmaxf(fmax3(pm[0], pm[1], pm[2]), pm[3]);
        const float m_new = fmaxf(m_run, mx * sl2);
        // The decision is made per warp (any lane over the threshold moves the
        // whole warp's maxima), because the TMEM accesses below must be
        // executed by all 32 lanes together; moving a maximum that grew by
        // less is exact all the same.
        if (__any_sync(0xffffffffu, m_new > m_run + kRescaleThreshold)) {
          if (j > jb) {
            // a row that has seen no key yet (window) has nothing to rescale
            const float alpha = (MASK == kMaskWindow && m_run == -INFINITY) ? 0.f : ex2(m_run - m_new);
            l_run *= alpha;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              uint32_t ov[32];
              tmem_ld32(tO + c, ov);
              tmem_wait_ld();
              reg_fence<32>(ov);
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
              tmem_st32(tO + c, ov);
            }
          }
          m_run = m_new;
        }
        // s * scale * log2(e) - m two columns per instruction, and the row sum
        // kept as two paired partial sums
        // (under a window a row may not have seen any key yet: its maximum is
        // still -inf, and every score of the block is -inf too)
        const float neg_m = (MASK == kMaskWindow && m_run == -INFINITY) ? 0.f : -m_run;
        const uint64_t sc2 = f32x2(sl2, sl2), nm2 = f32x2(neg_m, neg_m);
        uint64_t ps2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
        uint32_t pk[BN / 2];
#pragma unroll
        for (int c = 0; c < BN; c += 2) {
          float x0, x1;
          f32x2_split(ffma2(f32x2(s[c], s[c + 1]), sc2, nm2), x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          ps2[(c / 2) & 1] = fadd2(ps2[(c / 2) & 1], f32x2(p0, p1));
          pk[c / 2] = pack_bf16(p0, p1);
        }
        {
          float a0, a1, b0, b1;
          f32x2_split(ps2[0], a0, a1);
          f32x2_split(ps2[1], b0, b1);
          l_run += (a0 + a1) + (b0 + b1);
        }
        tmem_st32(tS + 0, pk);
        tmem_st32(tS + 32, pk + 32);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[t]);
      }
      // hand the row statistics to the epilogue
      if (!mbar_wait(&bars->st_empty[t], st_phase ^ 1, ab)) goto done;
      st_phase ^= 1;
      bars->stat_m[t][row] = m_run;
      bars->stat_l[t][row] = l_run;
      mbar_arrive(&bars->st_full[t]);
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ epilogue
    setmaxnreg_dec<RegSplit<MASK>::kEpilogue>();
    const int row = threadIdx.x & 127;
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t tph0 = 0, tph1 = 0, sf_ph = 0, sr_ph = 0;  // o_full / st_full phase of each tile
    const uint32_t stage32 = smem_u32(smem + C::OFF_STG);
    for (uint32_t it = 0;; ++it) {
      const int ui = sched_pop(bars, it, ab, true);
      if (ui == -2) goto done;
      if (ui < 0) break;
      const Unit u = decode<MASK>(p, ui);
      for (int t = 0; t < u.nt; ++t) {
        const uint32_t phase = t == 0 ? tph0 : tph1;
        if (t == 0)
          tph0 ^= 1;
        else
          tph1 ^= 1;
        if (!mbar_wait(&bars->o_full[t], phase, ab)) goto done;
        if (!mbar_wait(&bars->st_full[t], phase, ab)) goto done;
        tc_fence_after();
        const float m_fin = bars->stat_m[t][row];
        const float l_fin = bars->stat_l[t][row];
        mbar_arrive(&bars->st_empty[t]);
        const int qi = 2 * BM * u.m + BM * t + row;
        const bool valid = qi < u.rows;
        // A tile of 128 valid rows leaves through the staging box and TMA stores
        // (a warp store instruction would otherwise touch 32 rows); a tail tile is
        // written row by row, so no row past the end is touched.
        const bool full_tile = 2 * BM * u.m + BM * t + BM <= u.rows;
        const int orow = u.o_row0 + BM * t + row;
        const float inv_l = 1.0f / l_fin;
        __nv_bfloat16* dst = p.o + (static_cast<size_t>(orow) * p.H + u.h) * D;
        const uint32_t tO = tmem + lane_addr + 256 + t * 128;
#pragma unroll 1
        for (int rnd = 0; rnd < D / 64; ++rnd) {
          if (full_tile) {  // the box is free once TMA has read the previous one
            if (threadIdx.x == 256) {
              bulk_wait_read_all();
              mbar_arrive(&bars->ostg_free);
            }
            if (!mbar_wait(&bars->ostg_free, sf_ph, ab)) goto done;
            sf_ph ^= 1;
          }
#pragma unroll 1
          for (int q4 = 0; q4 < 4; ++q4) {  // 16 columns at a time
            const int c = 64 * rnd + 16 * q4;
            uint32_t ov[16];
            tmem_ld16(tO + c, ov);
            tmem_wait_ld();
            reg_fence<16>(ov);
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              pk[i] = pack_bf16(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l);
            if (full_tile) {
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                const uint32_t addr = stage32 + row * 128 + (((2 * q4 + i) ^ (row & 7)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * i]),
                             "r"(pk[4 * i + 1]), "r"(pk[4 * i + 2]), "r"(pk[4 * i + 3])
                             : "memory");
              }
            } else if (valid) {
#pragma unroll
              for (int i = 0; i < 2; ++i)
                st_global_v4(dst + c + 8 * i, pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            }
          }
          if (rnd == D / 64 - 1) {  // all of O is out of TMEM
            tc_fence_before();
            mbar_arrive(&bars->o_empty[t]);
          }
          if (full_tile) {
            fence_proxy_async_smem();
            mbar_arrive(&bars->ostg_full);
            if (!mbar_wait(&bars->ostg_full, sr_ph, ab)) goto done;
            sr_ph ^= 1;
            if (threadIdx.x == 256) {
              tma_store_2d(&tm_o, smem + C::OFF_STG, u.h * D + 64 * rnd, u.o_row0 + BM * t);
              bulk_commit_group();
            }
          }
        }
        if (valid && p.lse != nullptr)
          p.lse[static_cast<size_t>(u.h) * p.o_rows + orow] = (m_fin + log2f(l_fin)) * 0.69314718055994531f;
      }
    }
    if (threadIdx.x == 256) bulk_wait_all();  // every store has landed before the CTA exits
  } else {
    setmaxnreg_dec<RegSplit<MASK>::kIssue>();
    if (warp == 12 && lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t idesc_s = idesc_bf16(BM, BN, 0, 0);
      const uint32_t idesc_o = idesc_bf16(BM, D, 0, 1);
      const uint32_t sq = smem_u32(sQ), skv = smem_u32(sKV);
      uint32_t kv_it = 0;
      uint32_t p_phase[2] = {0, 0};
      uint32_t q_ph[2] = {0, 0};   // q_full parity of each tile's next load
      uint32_t o_cnt[2] = {0, 0};  // units that have used each O accumulator
      bool s0_early = false;       // the current unit's first S0 was issued during the previous unit
      auto stage_of = [&](uint32_t it) { return it % C::NSTAGE; };
      auto phase_of = [&](uint32_t it) { return (it / C::NSTAGE) & 1; };
      // Descriptors are formed once per GEMM and stepped through the K slices by
      // adding to their start-address field (address / 16, which stays inside
      // its 14 bits for any shared-memory address), keeping the issuing thread's
      // register use low.
      auto issue_s = [&](int t, uint32_t stage) {
        uint64_t qd = sdesc_sw128(sq + t * C::TILE_BYTES, 16, 1024);
        uint64_t kd = sdesc_sw128(skv + stage * C::TILE_BYTES, 16, 1024);
        asm volatile("" : "+l"(qd), "+l"(kd));  // formed here, not hoisted out of the unit loop
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off16 = ((k >> 2) * C::CHUNK_BYTES + (k & 3) * 32) >> 4;
          mma_ss(tmem + t * BN, qd + off16, kd + off16, idesc_s, k > 0);
        }
      };
      auto issue_pv = [&](int t, uint32_t stage, bool acc) {
        uint64_t vd = sdesc_sw128(skv + stage * C::TILE_BYTES, C::CHUNK_BYTES, 1024);
        asm volatile("" : "+l"(vd));
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_ts(tmem + 256 + t * 128, tmem + t * BN + k * 8, vd + ((k * 2048) >> 4), idesc_o,
                 (acc || k > 0) ? 1u : 0u);
      };
      // Once tile 0 of the current unit is done, the next unit's first score
      // GEMM (its tile-0 Q against its first K block) can run while tile 1's last
      // softmax does, so the tensor core does not idle at the unit boundary.  It
      // is issued only if the loader has already published that unit and its Q
      // tile and K block have landed (non-blocking checks: a blocking wait here
      // could hold up the releases the loader is waiting for); otherwise the next
      // unit starts as usual.  S0's TMEM columns are free: their P was read by
      // the tile's last PV, issued before (MMAs run in issue order).
      auto try_early_s0 = [&](uint32_t sched_it, uint32_t kv_next) {
        if (s0_early) return;
        const int slot = sched_it & 3;
        if (!mbar_try_wait(&bars->sched_full[slot], (sched_it >> 2) & 1)) return;
        if (*reinterpret_cast<volatile int*>(&bars->sched_unit[slot]) < 0) return;
        if (!mbar_try_wait(&bars->q_full[0], q_ph[0])) return;
        if (!mbar_try_wait(&bars->kv_full[stage_of(kv_next)], phase_of(kv_next))) return;
        tc_fence_after();
        issue_s(0, stage_of(kv_next));
        mma_commit(&bars->s_full[0]);
        s0_early = true;
      };
      if constexpr (MASK == kMaskNone || MASK == kMaskCausal) {
        // every query tile starts at block 0 and tile 0 may stop one block early:
        // the loop as measured fastest for these two
        for (uint32_t it = 0;; ++it) {
          const int ui = sched_pop(bars, it, ab, false);
          if (ui < 0) break;
          const Unit u = decode<MASK>(p, ui);
          const uint32_t kv_next = kv_it + 2 * u.n_kv;  // the next unit's first K block in the ring
          uint32_t ks = stage_of(kv_it);
          if (!mbar_wait(&bars->kv_full[ks], phase_of(kv_it), ab)) goto mma_done;
          if (!s0_early) {
            if (!mbar_wait(&bars->q_full[0], q_ph[0], ab)) goto mma_done;
            tc_fence_after();
            issue_s(0, ks);
            mma_commit(&bars->s_full[0]);
          }
          q_ph[0] ^= 1;
          s0_early = false;
          if (u.nt == 2) {
            if (!mbar_wait(&bars->q_full[1], q_ph[1], ab)) goto mma_done;
            q_ph[1] ^= 1;
            tc_fence_after();
            issue_s(1, ks);
            mma_commit(&bars->s_full[1]);
          }
          mma_commit(&bars->kv_empty[ks]);
          if (u.n_kv == 1) mma_commit(&bars->q_empty);
          ++kv_it;
          for (int j = 0; j < u.n_kv; ++j) {
            const uint32_t vs = stage_of(kv_it);
            if (!mbar_wait(&bars->kv_full[vs], phase_of(kv_it), ab)) goto mma_done;
            ++kv_it;
            const bool more = j + 1 < u.n_kv;
            uint32_t ks2 = 0;
            if (more) {  // K_{j+1}
              ks2 = stage_of(kv_it);
              if (!mbar_wait(&bars->kv_full[ks2], phase_of(kv_it), ab)) goto mma_done;
              ++kv_it;
            }
            // tile 0: O0 += P0 V_j, then S0 = Q0 K_{j+1}^T (tile 0 may stop one block early;
            // a single-tile unit visits every block with tile 0)
            if (j < u.je0) {
              if (j == 0) {
                if (!mbar_wait(&bars->o_empty[0], (o_cnt[0] & 1) ^ 1, ab)) goto mma_done;
                ++o_cnt[0];
              }
              if (!mbar_wait(&bars->p_full[0], p_phase[0], ab)) goto mma_done;
              p_phase[0] ^= 1;
              tc_fence_after();
              issue_pv(0, vs, j > 0);
              if (j + 1 == u.je0) {
                mma_commit(&bars->o_full[0]);
                if (u.nt == 1) mma_commit(&bars->kv_empty[vs]);
                try_early_s0(it + 1, kv_next);
              } else {
                issue_s(0, ks2);
                mma_commit(&bars->s_full[0]);
                if (u.nt == 1) {
                  mma_commit(&bars->kv_empty[vs]);
                  mma_commit(&bars->kv_empty[ks2]);
                  if (j + 2 == u.n_kv) mma_commit(&bars->q_empty);
                }
              }
            }
            if (u.nt == 1) continue;
            // tile 1: O1 += P1 V_j, then S1 = Q1 K_{j+1}^T
            if (j == 0) {
              if (!mbar_wait(&bars->o_empty[1], (o_cnt[1] & 1) ^ 1, ab)) goto mma_done;
              ++o_cnt[1];
            }
            if (!more) try_early_s0(it + 1, kv_next);  // a second chance before the last wait
            if (!mbar_wait(&bars->p_full[1], p_phase[1], ab)) goto mma_done;
            p_phase[1] ^= 1;
            tc_fence_after();
            issue_pv(1, vs, j > 0);
            mma_commit(&bars->kv_empty[vs]);
            if (!more) mma_commit(&bars->o_full[1]);
            if (more) {
              issue_s(1, ks2);
              mma_commit(&bars->s_full[1]);
              mma_commit(&bars->kv_empty[ks2]);
              if (j + 2 == u.n_kv) mma_commit(&bars->q_empty);
            }
          }
        }
      } else {
        // sliding window and block-sparse: each tile visits its own block range
        for (uint32_t it = 0;; ++it) {
          const int ui = sched_pop(bars, it, ab, false);
          if (ui < 0) break;
          const Unit u = decode<MASK>(p, ui);
          const uint32_t kv_next = kv_it + 2 * u.n_kv;  // the next unit's first K block in the ring
          const int j1 = u.j0 + u.n_kv;                 // blocks j0 .. j1-1 are in the ring, K then V
          const int jb1 = u.nt == 2 ? u.jb1 : j1, je1 = u.nt == 2 ? u.je1 : j1;  // tile 1's blocks
          // score GEMMs still to issue for this unit; Q is free once they are
          int s_left = (u.je0 - u.j0) + (je1 - jb1);
          auto s_issued = [&]() {
            if (--s_left == 0) mma_commit(&bars->q_empty);
          };
          uint32_t ks = stage_of(kv_it);
          if (!mbar_wait(&bars->kv_full[ks], phase_of(kv_it), ab)) goto mma_done;
          if (!s0_early) {
            if (!mbar_wait(&bars->q_full[0], q_ph[0], ab)) goto mma_done;
            tc_fence_after();
            issue_s(0, ks);
            mma_commit(&bars->s_full[0]);
          }
          q_ph[0] ^= 1;
          s0_early = false;
          if (u.nt == 2) {
            if (!mbar_wait(&bars->q_full[1], q_ph[1], ab)) goto mma_done;
            q_ph[1] ^= 1;
            tc_fence_after();
          }
          if (jb1 == u.j0) {
            issue_s(1, ks);
            mma_commit(&bars->s_full[1]);
            s_issued();
          }
          mma_commit(&bars->kv_empty[ks]);
          s_issued();  // tile 0's first S
          ++kv_it;
          for (int j = u.j0; j < j1; ++j) {
            const uint32_t vs = stage_of(kv_it);
            if (!mbar_wait(&bars->kv_full[vs], phase_of(kv_it), ab)) goto mma_done;
            ++kv_it;
            const bool more = j + 1 < j1;
            uint32_t ks2 = 0;
            if (more) {  // K_{j+1}
              ks2 = stage_of(kv_it);
              if (!mbar_wait(&bars->kv_full[ks2], phase_of(kv_it), ab)) goto mma_done;
              ++kv_it;
            }
            const bool t1_now = jb1 <= j && j < je1, t1_next = more && jb1 <= j + 1 && j + 1 < je1;
            // tile 0: O0 += P0 V_j, then S0 = Q0 K_{j+1}^T (tile 0 may stop early)
            if (j < u.je0) {
              if (j == u.j0) {
                if (!mbar_wait(&bars->o_empty[0], (o_cnt[0] & 1) ^ 1, ab)) goto mma_done;
                ++o_cnt[0];
              }
              if (!mbar_wait(&bars->p_full[0], p_phase[0], ab)) goto mma_done;
              p_phase[0] ^= 1;
              tc_fence_after();
              issue_pv(0, vs, j > u.j0);
              if (j + 1 == u.je0) {
                mma_commit(&bars->o_full[0]);
                if (!t1_now) mma_commit(&bars->kv_empty[vs]);
                try_early_s0(it + 1, kv_next);
              } else {
                issue_s(0, ks2);
                mma_commit(&bars->s_full[0]);
                s_issued();
                if (!t1_now) mma_commit(&bars->kv_empty[vs]);
                if (!t1_next) mma_commit(&bars->kv_empty[ks2]);
              }
            }
            // tile 1: O1 += P1 V_j, then S1 = Q1 K_{j+1}^T
            if (t1_now) {
              if (j == jb1) {
                if (!mbar_wait(&bars->o_empty[1], (o_cnt[1] & 1) ^ 1, ab)) goto mma_done;
                ++o_cnt[1];
              }
              if (!more) try_early_s0(it + 1, kv_next);  // a second chance before the last wait
              if (!mbar_wait(&bars->p_full[1], p_phase[1], ab)) goto mma_done;
              p_phase[1] ^= 1;
              tc_fence_after();
              issue_pv(1, vs, j > jb1);
              mma_commit(&bars->kv_empty[vs]);
              if (j + 1 == je1) mma_commit(&bars->o_full[1]);
            }
            if (t1_next) {
              issue_s(1, ks2);
              mma_commit(&bars->s_full[1]);
              s_issued();
              mma_commit(&bars->kv_empty[ks2]);
            }
            // (the two tiles' block ranges overlap or touch, so every block has a
            // reader; the releases below only guard the ring against a gap)
            if (j >= u.je0 && !t1_now) mma_commit(&bars->kv_empty[vs]);
            if (more && j + 1 >= u.je0 && !t1_next) mma_commit(&bars->kv_empty[ks2]);
          }
        }
      }
    mma_done:
      // wait until every issued MMA has landed before TMEM is released
      mma_commit(&bars->drain);
      {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&bars->drain, 0) && global_timer_ns() - t0 < kWaitTimeoutNs) {
        }
      }
    } else if (warp == 13 && lane == 0) {
      // ------------------------------------------------------------ TMA loader + scheduler
      // Static plan: this CTA's slice of the list.  Cluster Launch Control: the
      // CTA starts with its own index and, while loading a unit, asks the
      // hardware for a CTA that has not launched yet and takes over its unit
      // (aixai.ru summary, "Tile balancing and Cluster Launch Control").
      uint32_t kv_it = 0, u_phase = 0;
      int cur = p.use_clc ? static_cast<int>(blockIdx.x) : (u_begin < u_end ? u_begin : -1);
      for (uint32_t it = 0;; ++it) {
        const int slot = it & 3;
        if (!mbar_wait(&bars->sched_empty[slot], ((it >> 2) & 1) ^ 1, ab)) break;
        bars->sched_unit[slot] = cur;
        mbar_arrive(&bars->sched_full[slot]);
        if (cur < 0) break;
        if (p.use_clc) {
          mbar_expect_tx(&bars->clc_bar, 16);
          clc_try_cancel(&bars->clc_resp, &bars->clc_bar);
        }
        const Unit u = decode<MASK>(p, cur);
        if (!mbar_wait(&bars->q_empty, u_phase ^ 1, ab)) break;
        for (int t = 0; t < u.nt; ++t) {
          mbar_expect_tx(&bars->q_full[t], C::TILE_BYTES);
#pragma unroll
          for (int c = 0; c < C::NCHUNK; ++c)
            tma_load_2d(&tm_q, &bars->q_full[t], sQ + t * C::TILE_BYTES + c * C::CHUNK_BYTES, u.h * D + c * 64,
                        u.q_row0 + BM * t);
        }
        bool ok = true;
        for (int j = 0; j < u.n_kv && ok; ++j) {
          for (int w = 0; w < 2; ++w) {
            const uint32_t s = kv_it % C::NSTAGE, ph = (kv_it / C::NSTAGE) & 1;
            if (!mbar_wait(&bars->kv_empty[s], ph ^ 1, ab)) {
              ok = false;
              break;
            }
            mbar_expect_tx(&bars->kv_full[s], C::TILE_BYTES);
            const CUtensorMap* tm = w == 0 ? &tm_k : &tm_v;
#pragma unroll
            for (int c = 0; c < C::NCHUNK; ++c)
              tma_load_2d(tm, &bars->kv_full[s], sKV + s * C::TILE_BYTES + c * C::CHUNK_BYTES, u.g * D + c * 64,
                          u.kv0 + BN * (MASK == kMaskTopK ? u.sel[j] : u.j0 + j));
            ++kv_it;
          }
        }
        if (!ok) break;
        u_phase ^= 1;
        int nxt;
        if (p.use_clc) {
          if (!mbar_wait(&bars->clc_bar, it & 1, ab)) break;
          nxt = clc_cancelled_x(&bars->clc_resp);
          if (nxt >= p.n_units) nxt = -1;
        } else {
          nxt = cur + 1 < u_end ? cur + 1 : -1;
        }
        cur = nxt;
      }
      if (*ab.flag) {
        // aborting: let copies already in flight land before the CTA exits
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

template <int D, int MASK>
int launch_impl(const FwdArgs& a) {
  using C = Cfg<D>;
  CUtensorMap tq, tk, tv;
  int st = make_map_2d(&tq, a.q, static_cast<uint64_t>(a.H) * D, a.q_rows, 64, BM);
  if (st == JFA_OK) st = make_map_2d(&tk, a.k, static_cast<uint64_t>(a.Hkv) * D, a.kv_rows, 64, BN);
  if (st == JFA_OK) st = make_map_2d(&tv, a.v, static_cast<uint64_t>(a.Hkv) * D, a.kv_rows, 64, BN);
  CUtensorMap to;  // O, for the epilogue's TMA stores of full tiles
  if (st == JFA_OK) st = make_map_2d(&to, a.o, static_cast<uint64_t>(a.H) * D, a.o_rows, 64, BM);
  if (st != JFA_OK) return st;
  auto kern = fwd_kernel<D, MASK>;
  static PerDeviceOnce setup;  // per instantiation
  st = setup.run([&]() -> int {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return JFA_ERR_CUDA;
    if (fa.numRegs * kThreads < RegSplit<MASK>::kTotal) return JFA_ERR_UNSUPPORTED;  // never granted otherwise
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC) != cudaSuccess)
      return JFA_ERR_CUDA;
    return JFA_OK;
  });
  if (st != JFA_OK) return st;
  Params p;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.offsets = a.offsets_dev;
  p.units = reinterpret_cast<const int4*>(a.units);
  p.cta_start = a.cta_start;
  p.err = a.err;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.nq = a.nq;
  p.o_rows = a.o_rows;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.n_units = a.n_units;
  p.use_clc = a.use_clc;
  p.win_left = a.win_left;
  p.win_right = a.win_right;
  p.topk_sel = a.topk_sel;
  p.topk_qb = a.topk_qb;
  p.topk = a.topk;
  ProfileScope prof(kKindFwd, a.stream);
  kern<<<a.use_clc ? a.n_units : a.n_cta, kThreads, C::SMEM_ALLOC, a.stream>>>(tq, tk, tv, to, p);
  return cudaGetLastError() == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

}  // namespace fwd

int launch_fwd(const FwdArgs& a) {
  if (a.D == 128) {
    if (a.mask == kMaskWindow) return fwd::launch_impl<128, kMaskWindow>(a);
    if (a.mask == kMaskTopK) return fwd::launch_impl<128, kMaskTopK>(a);
    return a.mask == kMaskCausal ? fwd::launch_impl<128, kMaskCausal>(a) : fwd::launch_impl<128, kMaskNone>(a);
  }
  if (a.mask == kMaskWindow) return fwd::launch_impl<64, kMaskWindow>(a);
  if (a.mask == kMaskTopK) return fwd::launch_impl<64, kMaskTopK>(a);
  return a.mask == kMaskCausal ? fwd::launch_impl<64, kMaskCausal>(a) : fwd::launch_impl<64, kMaskNone>(a);
}

}  // namespace jfa
