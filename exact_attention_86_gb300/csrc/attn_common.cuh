// Definitions shared by the translation units of the attention library:
// the launch parameters, the work-unit order, the bounded waits and the
// per-unit queue of the persistent kernels.  Each translation unit gets its
// own device status word (g_attn_status, in its anonymous namespace); the
// library's attn_check_device_status reads and clears all of them.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn.h"
#include "sm103_ptx.cuh"

namespace attn_detail {

using namespace attn_sm103;

constexpr int kBQ = 128;          // query rows per work unit (MMA M, TMEM lanes)
constexpr int kBK = 128;          // keys per K/V tile (MMA N of QK^T)
constexpr int kThreads = 384;
// Register split (setmaxnreg): the block launches at 168 per thread; warpgroup 2
// (producer, issuers) drops to 104 and the two softmax warpgroups rise to 200:
//   384 x 168 = 64512 = 256 x 200 + 128 x 104; per SM sub-partition
//   (one warp of each warpgroup) (200 + 200 + 104) x 32 <= 16384.
constexpr int kRegsSoftmax = 200;
constexpr int kRegsOther = 104;
constexpr int kSoftmaxWarps = 8;
constexpr int kWarpLoad = 8;
constexpr int kWarpQK = 9;
constexpr int kWarpPV = 10;
constexpr int kWarpLoadV = 11;   // forward: the V producer
constexpr int kUnitQ = 4;           // depth of a CTA's unit queue
constexpr int kUnitQReaders = 10;   // warps that read it: QK^T and P V issuers, 8 softmax warps (+ the V producer with split rings)
constexpr float kLn2 = 0.69314718055994530942f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: far above any legitimate wait
constexpr uint64_t kDrainLimitNs = 100000000ull;   // 0.1 s for draining after an abort

enum WaitSite : uint32_t {
  kSiteQEmpty = 1,
  kSiteKvEmpty = 2,
  kSiteQFull = 3,
  kSiteKvFull = 4,
  kSitePFull = 5,
  kSiteSFull = 6,
  kSiteOFull = 7,
  kSiteSelftest = 8,
  kSiteSFree = 9,
  kSitePFree = 10,
  kSiteUnitQ = 11,
  kSiteAlign = 12,   // not a wait: the block's shared memory was not 1024-byte aligned
  kSitePvIssued = 13,
};

// Division by a divisor fixed for a launch, with one multiply-high, an add
// and a shift (the method of Granlund and Montgomery, "Division by invariant
// integers using multiplication", 1994): for d >= 1 let s = ceil(log2 d) and
// m = floor(2^32 (2^s - d) / d) + 1; then floor(n / d) = (mulhi(n, m) + n) >> s
// for every 0 <= n < 2^31 (the sum stays below 2^32).  The work-unit decode of
// every role used to spend most of its time in general integer divisions.
struct FastDiv {
  uint32_t d, m, s;
  __device__ __forceinline__ int div(int n) const {
    return static_cast<int>((__umulhi(static_cast<uint32_t>(n), m) + static_cast<uint32_t>(n)) >> s);
  }
};

struct Params {
  uint16_t* o;
  float* lse;
  const int32_t* kv_lens;
  int B, H, Sq, Sk;
  int n_qtiles;
  int head_group;          // causal order: heads per group (their K/V fit in a share of L2)
  int num_splits;          // key ranges per (b, h, query tile); 1 = whole rows
  int total_units;
  float* o_part;           // split mode: fp32 [num_splits][B*H*Sq][D] normalised partial outputs
  float* lse_part;         //             fp32 [num_splits][B*H*Sq] partial LSE; nullptr = write o/lse
  // packed variable-length mode (cu_q != nullptr): q/o [total_q, H, D], k/v
  // [total_k, H, D], lse [H, total_q]; sequence b owns query tokens
  // [cu_q[b], cu_q[b+1]) and key tokens [cu_k[b], cu_k[b+1]); B = batch and
  // Sq = the largest query length (it sizes the grid)
  const int32_t* cu_q;
  const int32_t* cu_k;
  int total_q, total_k;
  // paged-KV mode (block_table != nullptr, with packed queries): k/v caches
  // [num_pages, page_size, H, D]; key j of sequence b is slot j % page_size of
  // page block_table[b * max_pages + j / page_size]; seqlens_k[b] keys
  const int32_t* block_table;
  const int32_t* seqlens_k;
  int page_size, max_pages, num_pages;
  int cache_tokens;        // num_pages * page_size: a key coordinate that reads zeros
  uint32_t* sched;         // dynamic scheduling: [0] next unit to claim, [1] CTAs done (both 0 on entry
                           // and on exit); nullptr: static round-robin
  float c;                 // |scale| * log2(e) (E4M3: |scale * q_descale * k_descale| * log2(e))
  float v_scale;           // 1, or the E4M3 V descale (multiplies O)
  uint32_t idesc_qk;       // negate-A set when scale < 0
  uint32_t idesc_pv;
  uint64_t wait_limit_ns;
  // divisors of the unit decode, set at launch (with_divisors)
  FastDiv fd_splits, fd_qtiles, fd_group_units, fd_group_heads, fd_last_heads, fd_H, fd_grid;
  int last_group;          // causal order: index of the last head group (it may hold fewer heads)
  // Self test of the give-up path only (attn_selftest_fwd_abort): block 0's
  // producer leaves out its K fill with this index, so the bounded wait of the
  // fill's consumer must give up and every role must drain; -1 otherwise.
  int selftest_skip_fill = -1;
  // E4M3 only: V given in rows, [B, H, Sk, D] (the P V product then reads it
  // MN-major, like bf16 V); 0: V given transposed, [B, H, D, Sk] (K-major)
  int v_rows = 0;
  int o_align32 = 0;       // o is 32-byte aligned: the epilogue writes 32-byte pieces
};


// Lazy rescale threshold (log2 units) and the shift of P (log2 units): each P
// term is 2^(x - m + shift) <= 2^(tau + shift).  bf16 P: tau 16, shift 0.
// E4M3 P (largest finite value 448): tau 4.5, shift 4, so terms stay <= 2^8.5
// and terms down to 2^-13 of the reference keep a nonzero code.
template <bool FP8>
struct Prec {
  static constexpr float kTau = FP8 ? 4.5f : 16.0f;
  static constexpr float kShift = FP8 ? 4.0f : 0.0f;
  static constexpr float kSumLimit = FP8 ? 362.03867196751236f : 65536.0f;  // 2^(kTau + kShift)
};
// ---------------------------------------------------------------- host side

inline FastDiv make_fastdiv(int divisor) {
  FastDiv f;
  f.d = static_cast<uint32_t>(divisor < 1 ? 1 : divisor);
  uint32_t sh = 0;
  while ((1ull << sh) < f.d) ++sh;
  f.s = sh;
  f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << sh) - f.d)) / f.d + 1);
  return f;
}

// The launch's Params with the divisors of the unit decode filled in (grid:
// the number of blocks the kernel is launched with).
inline Params with_divisors(const Params& p0, int grid) {
  Params p = p0;
  const int bh = p.B * p.H;
  const int hg = p.head_group < 1 ? 1 : p.head_group;
  const int groups = bh > 0 ? (bh + hg - 1) / hg : 1;
  p.fd_splits = make_fastdiv(p.num_splits);
  p.fd_qtiles = make_fastdiv(p.n_qtiles);
  p.fd_group_units = make_fastdiv(hg * p.n_qtiles);
  p.fd_group_heads = make_fastdiv(hg);
  p.last_group = groups - 1;
  p.fd_last_heads = make_fastdiv(bh - (groups - 1) * hg);
  p.fd_H = make_fastdiv(p.H);
  p.fd_grid = make_fastdiv(grid);
  p.o_align32 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0 ? 1 : 0;
  return p;
}

}  // namespace attn_detail

namespace {

using namespace attn_detail;
using namespace attn_sm103;

// [0]: 1 once any wait gave up; [1]: site of the first one; [2]: its block.
__device__ uint32_t g_attn_status[3];

// Unit processed at the t-th step of the persistent loop (t = blockIdx.x +
// k * gridDim.x).  Causal units come longest first; they are dealt to the CTAs
// in alternating direction each round ("snake" order), which evens out the
// per-CTA sums of their lengths.  Values >= total_units are skipped.
template <bool CAUSAL>
__device__ __forceinline__ int unit_at(const Params& p, int t) {
  if (!CAUSAL) return t;
  const int round = p.fd_grid.div(t);
  const int pos = t - round * static_cast<int>(gridDim.x);
  return (round & 1) ? round * static_cast<int>(gridDim.x) + (static_cast<int>(gridDim.x) - 1 - pos) : t;
}

__device__ __noinline__ void record_give_up(uint32_t site) {
  if (atomicCAS(&g_attn_status[1], 0u, site) == 0u) g_attn_status[2] = blockIdx.x;
  atomicOr(&g_attn_status[0], 1u);
  __threadfence();
}

// Bounded wait for the phase of `bar` with parity `parity`.  Returns false when
// the CTA is aborting or the limit passed (then the give-up is recorded).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint32_t site,
                                           uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0u) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        record_give_up(site);
        return false;
      }
    }
  }
}

// The same wait for a whole warp: every lane waits, and the outcome is made
// warp-uniform so that warp-collective operations after it never miss a lane.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint32_t site,
                                          uint64_t limit_ns) {
  return __all_sync(0xffffffffu, wait_phase(bar, parity, abort_flag, site, limit_ns));
}

// Next unit of this CTA from its unit queue, which the producer lane fills:
// every reading warp takes each entry once, in order.  Returns the unit, -1
// at the end of the CTA's work, or -2 when the wait gave up.
__device__ __forceinline__ int take_unit(uint32_t& k, volatile int* unit_q, uint32_t full0, uint32_t empty0,
                                         volatile int* abort_flag, uint64_t limit, int lane) {
  const uint32_t slot = k % kUnitQ;
  if (!wait_warp(full0 + 8 * slot, (k / kUnitQ) & 1u, abort_flag, kSiteUnitQ, limit)) return -2;
  const int unit = unit_q[slot];
  __syncwarp();
  if (lane == 0) mbar_arrive(empty0 + 8 * slot);
  ++k;
  return unit;
}

// Wait used only while draining after an abort: ignores the abort flag.
__device__ __forceinline__ void wait_phase_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kDrainLimitNs) return;
  }
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

// One warp's arrival on a barrier that counts warps: every lane's tcgen05
// traffic is ordered before the warp synchronisation, then one lane arrives.
__device__ __forceinline__ void warp_arrive_after_tc(uint32_t bar, int lane) {
  tc_fence_before_sync();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

}  // namespace
