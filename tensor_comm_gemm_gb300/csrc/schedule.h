// Host-side schedule model shared by the two AG entry points (no device code).
#pragma once

#include "tpo_params.h"

namespace tpo {

// Producer CTAs set aside when the automatic column plan sizes an AG launch's
// GEMM grid (the schedule model's largest producer count).
constexpr int AUTO_COLS_PRODUCERS = 32;

// The automatic column plan (option col_split 0): the fewest column tiles of
// at most 256 columns, unless the launch has at most half as many tiles as it
// can have GEMM CTA groups (gemm_groups).  Then every group's 32-column strips
// are split into more, narrower tiles (down to one strip each) while all of
// them still fit in one round: a tile's K loop costs about the same at any
// width, so the round takes as long, and each tile's epilogue (its share of
// the output to convert and store) is shorter.  Sets p's column tiling.
void auto_columns(Params& p, long long m, int gemm_groups);

// The host schedule model's producer CTA count for an overlapped AG launch
// with default options, whose tiles (uniform column tiles), K blocks and chunk
// size p describes, on num_sms SMs with max_pairs co-resident CTA pairs
// (ctx.cu; the entry point without a context uses it).
int model_producers(const Params& p, int cg, int tp, int num_sms, int max_pairs);

}  // namespace tpo
