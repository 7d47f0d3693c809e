// Host entry points of the two-query-tile forward kernel (attn_fwd_pair.cu),
// a translation unit of its own so that its code leaves the register
// allocation of attn_fwd.cu's kernels untouched.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn.h"

// 1: causal padded batches also take the two-tile kernel (a build option; the
// causal instantiations are compiled only then)
#ifndef ATTN_PAIR_CAUSAL
#define ATTN_PAIR_CAUSAL 0
#endif

namespace attn_detail {
struct Params;
}

namespace attn_pair_host {

// Launches the padded forward over units of two 128-row query tiles
// (p.n_qtiles = tile pairs per head, p.total_units = B * H * pairs; every
// other field as for attn_fwd_kernel, without key ranges) on `stream`, with
// one block per SM up to the number of units.
attn_status launch(int D, bool causal, int num_sms, const CUtensorMap& mq, const CUtensorMap& mk,
                   const CUtensorMap& mv, const attn_detail::Params& p, cudaStream_t stream);

// Reads this translation unit's device status word into host[3] ([0]: a wait
// gave up, [1]: its site, [2]: its block) and clears it if it was set.
attn_status status_read_clear(uint32_t host[3]);

}  // namespace attn_pair_host
