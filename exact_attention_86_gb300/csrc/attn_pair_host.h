// Host entry points of the two-query-tile forward kernel (attn_fwd_pair.cu),
// a translation unit of its own so that its code leaves the register
// allocation of attn_fwd.cu's kernels untouched.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn.h"

namespace attn_detail {
struct Params;
}

namespace attn_pair_host {

// Whether a padded batch of B x H heads (Sq queries, Sk keys, head dimension
// D; bf16, or E4M3 when fp8) runs faster on the two-tile kernel than on the
// one-tile kernel of attn_fwd.cu, on a device with num_sms SMs.  A cost model
// of each work unit, host arithmetic only; false for arguments out of range.
bool use_pair(int B, int H, int Sq, int Sk, int D, bool causal, int num_sms, bool fp8);

// Launches the forward over units of two 128-row query tiles (p.n_qtiles =
// tile pairs per head, p.total_units = B * H * pairs; every other field as
// for attn_fwd_kernel, without key ranges; fp8: E4M3 inputs, with the tensor
// maps, descriptors and descales attn_fwd_fp8_ex builds; p.cu_q set: a packed
// or paged bf16 batch, with attn_fwd_varlen's or attn_fwd_paged's maps and
// fields, p.sched its optional counter) on `stream`, with one block per SM up
// to the number of units.  Padded causal batches get a static longest-first
// deal of their units (see build_schedule); packed batches claim their units
// from p.sched when it is set; the rest take the round-robin deal.
attn_status launch(int D, bool causal, bool fp8, int num_sms, const CUtensorMap& mq, const CUtensorMap& mk,
                   const CUtensorMap& mv, const attn_detail::Params& p, cudaStream_t stream);

// The static deal of a causal batch's pair units to `grid` blocks, in the
// kernel's unit order (head groups of `head_group` heads, longest units first
// within a group): owner[t] is the block that runs unit t.  Each unit in
// turn goes to the block with the least modelled work so far (the lowest
// index among equals).  Returns the number of units (B * H * pairs), or -1
// when it exceeds max_units or an argument is out of range (owner untouched).
int64_t build_schedule(int B, int H, int Sq, int Sk, int head_group, int grid, uint8_t* owner, int64_t max_units);

// Reads this translation unit's device status word into host[3] ([0]: a wait
// gave up, [1]: its site, [2]: its block) and clears it if it was set.
attn_status status_read_clear(uint32_t host[3]);

}  // namespace attn_pair_host
