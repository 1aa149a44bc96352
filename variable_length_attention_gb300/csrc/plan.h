// plan.h -- host planners shared by the API layer (see plan.cpp).
#pragma once
#include <cstdint>
#include <vector>

namespace jfa {

constexpr int kFwdRows = 256;  // query rows per forward unit (two 128-row tiles)
constexpr int kKvBlock = 128;  // keys per K/V block
constexpr int kBlk = 64;       // block-diagonal block size

// JFA_OK, or the status describing what is wrong with the offsets
// (max_len < 0 skips the length bound).
int check_offsets(const int32_t* offsets, int batch, int max_len);

// Each returns the unit count; lists are CTA-major int32 quadruples.
int plan_fwd(const int32_t* offsets, int batch, int H, int nq, int causal, int n_cta, std::vector<int32_t>* units,
             std::vector<int32_t>* cta_start);
int plan_bwd(const int32_t* offsets, int batch, int H, int nq, int causal, int n_cta, std::vector<int32_t>* units,
             std::vector<int32_t>* cta_start);
// The same under a window: query i sees keys [i - left, i + right] of its
// sequence (a negative bound leaves its side open; causal is (-1, 0)).
int plan_fwd_window(const int32_t* offsets, int batch, int H, int nq, int left, int right, int n_cta,
                    std::vector<int32_t>* units, std::vector<int32_t>* cta_start);
int plan_bwd_window(const int32_t* offsets, int batch, int H, int nq, int left, int right, int n_cta,
                    std::vector<int32_t>* units, std::vector<int32_t>* cta_start);
// Block-sparse forward: the forward's units, each costing the blocks it visits
// (min(topk, key blocks of its sequence)).
int plan_fwd_topk(const int32_t* offsets, int batch, int H, int nq, int topk, int n_cta, std::vector<int32_t>* units,
                  std::vector<int32_t>* cta_start);
// The device copy of a unit list: each entry's fourth field (the cost the
// planner sorted by) replaced by the length of the entry's sequence, so that a
// kernel decoding a unit has it without a second load that depends on the first.
void units_for_device(std::vector<int32_t>* units, const int32_t* offsets);
// Returns the number of programs P.
int plan_block(const int32_t* offsets, int batch, int H, int n_sm, std::vector<int32_t>* bpb,
               std::vector<int32_t>* prog_start);

}  // namespace jfa
