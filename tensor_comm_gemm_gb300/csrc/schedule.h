// Host-side schedule model shared by the two AG entry points (no device code).
#pragma once

#include "tpo_params.h"

namespace tpo {

// The host schedule model's producer CTA count for an overlapped AG launch
// with default options, whose tiles (uniform column tiles), K blocks and chunk
// size p describes, on num_sms SMs with max_pairs co-resident CTA pairs
// (ctx.cu; the entry point without a context uses it).
int model_producers(const Params& p, int cg, int tp, int num_sms, int max_pairs);

}  // namespace tpo
