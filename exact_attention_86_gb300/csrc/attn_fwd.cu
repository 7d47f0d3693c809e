// Exact fused attention forward for GB300 (sm_103a).
//
// Computes O = softmax(scale * Q K^T + mask) V and LSE = ln(sum_j exp(scale * q.k_j))
// for a padded batch [B, H, S, D] of bf16 tensors ("Kernel Fusion and the Memory
// Wall", section "FlashAttention: avoid the full score matrix").  Each CTA owns
// one block of 128 query rows at a time and streams the K/V tiles of that head
// past it ("Attention softmax fusion", section "The tile loop"); the score tile
// lives only in Tensor Memory and registers, and the running max / sum /
// numerator are corrected by exp(m_old - m_new) whenever a later tile raises
// the row maximum (same section, second paragraph).  Nothing of size Sq x Sk is
// ever written to device memory.
//
// CTA layout (384 threads, persistent over work units):
//   warps 0-3  softmax, columns 0-63 of every score tile (one thread per row)
//   warps 4-7  softmax, columns 64-127 (the partner thread of the same row)
//   warp 8     TMA producer of the units, Q and the K ring (one lane)
//   warp 9     TMEM owner; issues S = Q K^T (whole warp, one elected lane)
//   warp 10    issues O += P V (whole warp, one elected lane)
//   warp 11    TMA producer of the V ring (one lane; split rings only, else idle)
//
// Tensor Memory (512 columns x 128 lanes, lane = query row):
//   [  0,128)  S buffer 0      [128,256)  S buffer 1     (fp32 scores)
//   [256,320)  P buffer 0      [320,384)  P buffer 1     (bf16 pairs)
//   [384,384+D) O accumulator (fp32)
// With two S buffers the QK^T of tile j+1 runs while the softmax of tile j
// works, and with P apart from S the PV of tile j runs while QK^T proceeds:
// the two issuing warps each feed one independent stream of MMAs.  One warp
// issues a 128x128x16 MMA no faster than about one per 110 cycles (measured),
// more than the 64 cycles the tensor core needs for it, so both streams must
// be in flight to keep the tensor pipe busy.
//
// Every mbarrier wait is bounded (global timer); a wait that gives up records
// the site in a device status word, raises a CTA-wide abort flag, and every
// role drains what it has in flight, frees TMEM and returns.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>

#include "attn.h"
#include "attn_common.cuh"
#include "attn_pair_host.h"
#include "sm103_ptx.cuh"

using namespace attn_sm103;

namespace {

// Fixed split-KV scratch of attn_fwd_splitkv_noalloc: a static device array,
// instantiated once in every device context that loads the library, so that
// entry point needs neither an allocation nor a caller workspace.
__device__ __align__(256) uint8_t g_splitkv_scratch[ATTN_SPLITKV_SCRATCH_BYTES];

#ifndef ATTN_SPLIT_SLOTS_K
#define ATTN_SPLIT_SLOTS_K 3   // K slots of the split rings at D = 128 (bf16)
#endif
#ifndef ATTN_SPLIT_SLOTS_V
#define ATTN_SPLIT_SLOTS_V 2   // V slots of the split rings at D = 128 (bf16)
#endif

template <int D, bool FP8 = false, bool SPLIT = false>
struct Geo {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kElem = FP8 ? 1 : 2;            // bytes per element of Q, K, V
  static constexpr int kRowBytes = D * kElem;          // one row of a Q or K tile (and of V in rows)
  static constexpr int kTileBytes = 128 * D * kElem;   // one Q, K or V tile (128 rows)
  // Rows of 128 bytes (bf16 D = 64, E4M3 D = 128) or 256 bytes (bf16 D = 128,
  // two 64-column chunks) use the 128-byte swizzle; the 64-byte rows of E4M3
  // at D = 64 the 64-byte swizzle (8-row atoms of 64 bytes, 512 bytes apart).
  static constexpr bool kSw64 = kRowBytes == 64;
  static constexpr int kChunkBytes = kSw64 ? 128 * 64 : 128 * 128;  // 128 rows of one swizzle column
  static constexpr int kChunks = kSw64 ? 1 : kRowBytes / 128;
  static constexpr int kChunkElems = kSw64 ? 64 : 128 / kElem;      // elements per row of a chunk
  static constexpr uint32_t kSwMode = kSw64 ? kSmemSwizzle64B : kSmemSwizzle128B;
  static constexpr uint32_t kSbo = kSw64 ? 512 : 1024;               // 8-row groups of a chunk
  static constexpr int kKSteps = D * kElem / 32;       // QK^T instructions: 32 B of D each
  // K and V tiles in shared memory.  Padded batches (one ring): as many as
  // the 227 KB a block may use leave after the control block, the exchange
  // buffers and Q.  Packed and paged batches (split rings) at D = 128: 3 K
  // and 2 V slots (measured faster than 3 + 3 there).
  static constexpr int kSlots =
      (D == 128 && !FP8) ? (SPLIT ? ATTN_SPLIT_SLOTS_K + ATTN_SPLIT_SLOTS_V : 6) : (kSw64 ? 16 : 12);
  // Two layouts of the K/V tiles over those slots (both modelled by the
  // protocol tests):
  //  single ring (padded batches): the producer fills K_0 V_0 K_1 V_1 ... in
  //    order, position pos = 2 t (+1 for V) in slot pos % kSlots.  With an odd
  //    depth a slot alternates between K and V fills, so each slot has one
  //    "full" barrier per kind (waited on, phase after phase, by the one issuer
  //    that consumes that kind: a parity wait can never match a phase two
  //    fills old) and one "empty" barrier counting all its fills.  A K fill
  //    then waits for the P V of an earlier tile, which paces the QK^T issuer
  //    (measured faster here than the split layout, 3 %).
  //  split rings (packed and paged batches): K_t in slot t % kSlotsK, V_t in
  //    slot kSlotsK + t % kSlotsV, each ring filled by its own producer warp,
  //    so a K fill never waits behind a V fill or its page lookups (measured
  //    faster there: paged 6 %, packed 2 %).
  static constexpr int kSlotsK = (D == 128 && !FP8 && SPLIT) ? ATTN_SPLIT_SLOTS_K : kSlots / 2;
  static constexpr int kSlotsV = kSlots - kSlotsK;
  struct Fill {
    uint32_t slot;       // shared-memory slot of the tile
    uint32_t full_use;   // phase index on the slot's full barrier of its kind
    uint32_t empty_use;  // phase index on the slot's empty barrier (fills of the slot before it)
  };
  // where K_t (is_v false) or V_t goes
  static __device__ __forceinline__ Fill fill_of(uint32_t t, bool is_v, bool split) {
    if (split) {
      const uint32_t n = is_v ? kSlotsV : kSlotsK;
      return {(is_v ? static_cast<uint32_t>(kSlotsK) : 0u) + t % n, t / n, t / n};
    }
    const uint32_t pos = 2 * t + (is_v ? 1u : 0u);
    return {pos % kSlots, (kSlots & 1) ? (pos / kSlots) >> 1 : pos / kSlots, pos / kSlots};
  }
  // Two TMEM protocols (both modelled by the protocol tests):
  //  bf16: S buffers 0/1 at [0,128) and [128,256), released by the softmax
  //        once read; P buffers 0/1 at [256,320) and [320,384); one O buffer
  //        at [384, 384 + D).
  //  E4M3 (kPInS): S buffers as above, P_b written over the S_b columns each
  //        half has read (half h: from column 64 h), so S_b is released by
  //        the P V commit; O buffers 0/1 at [256, 256 + D) and [256 + D,
  //        256 + 2 D), alternating between consecutive units.  With half-time
  //        products the shorter QK^T lead costs nothing and the P buffer wait
  //        disappears (measured faster for E4M3, slower for bf16).
  static constexpr bool kPInS = FP8;
  static constexpr int kOBufs = kPInS ? 2 : 1;
  static constexpr uint32_t kTmemS = 0;                  // + 128 * buffer
  static constexpr uint32_t kTmemP = 256;                // + 64 * buffer (bf16 protocol)
  static constexpr uint32_t kTmemO = kPInS ? 256 : 384;  // + D * buffer
  static constexpr int kTmemCols = 512;
  // TMEM column of the P operand of the kk-th P V instruction, relative to the
  // tile's S buffer (P over S) or P buffer (16 bf16 keys or 32 E4M3 keys = 8
  // columns per instruction)
  static __device__ __forceinline__ uint32_t p_col(int kk) {
    constexpr int per_half = FP8 ? 2 : 4;  // instructions per half's 64 keys
    if constexpr (kPInS)
      return 64u * static_cast<uint32_t>(kk / per_half) + 8u * static_cast<uint32_t>(kk % per_half);
    return 8u * static_cast<uint32_t>(kk);
  }
  // Control block [0, 1024), exchange buffers [1024, 3072), Q, the ring.  The
  // dynamic shared memory of a block starts 1024-byte aligned (checked at
  // kernel entry), as the 128-byte swizzle atoms need, so no slack is added.
  static constexpr int kOffQ = 3072;
  static constexpr int kOffRing = kOffQ + kTileBytes;
  // E4M3 at D = 64 leaves room to spare: an unused tile-sized pad after the
  // ring keeps any read of the last slot inside the allocation
  static constexpr int kPadBytes = kSw64 ? kTileBytes : 0;
  static constexpr int kSmemBytes = kOffRing + kSlots * kTileBytes + kPadBytes;
  static_assert(kOffQ % 1024 == 0 || kTileBytes % 1024 == 0, "swizzle atoms 1024-byte aligned");
  static_assert(kSmemBytes <= 232448, "shared memory per block");
  static_assert(kSlots <= 16, "barrier initialisation: one lane per slot among lanes 0-15");
};

struct Unit {
  int b, h, q0;            // q0: position of the unit's first query row within its sequence
  int rows;                // query rows of the unit that exist (<= 128; 0: nothing to do)
  int q_tok0, k_tok0;      // packed mode: token index of the first query row / first key
  int kv;                  // valid keys of this batch entry (kv_lens clamped to [0, Sk])
  int j0;                  // first K tile of the unit
  int n;                   // K tiles the unit processes (0: no valid key for any row)
  int split;               // key range index (split mode)
};

struct Ctrl {
  uint64_t q_full, q_empty;
  uint64_t k_full[16], v_full[16], kv_empty[16];  // per slot; full: one per kind (Geo::fill_of)
  uint64_t s_full[2], s_free[2], p_full[2], p_free[2];
  uint64_t o_full[2], o_free[2];
  uint64_t pv_issued;  // the P V issuer has issued the last product of a unit
  uint64_t uq_full[4], uq_empty[4];  // the CTA's unit queue (filled by the producer lane)
  int unit_q[4];
  uint64_t drain[2];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Ctrl) <= 1024, "control block");

// Exchange buffers (shared memory, after the control block at +1024):
// xmax[2][2][128] fp32 (tile parity, half, row).  The partial row sums of a
// unit's epilogue go through xmax[b ^ 1], b the parity of the unit's last tile:
// both halves of a row passed that tile's barrier after their last read of
// xmax[b ^ 1] (the tile before), and the next write to it is the next unit's
// first tile, after two more barriers of the pair.
struct Xchg {
  float xmax[2][2][kBQ];
};
static_assert(sizeof(Xchg) <= 2048, "exchange buffers");

template <bool CAUSAL>
__device__ __forceinline__ Unit decode_unit(const Params& p, int t_in) {
  Unit u;
  // split mode: the key tiles of a (b, h, query tile) are cut into num_splits
  // contiguous ranges, consecutive units
  const int t = p.fd_splits.div(t_in);
  u.split = t_in - t * p.num_splits;
  int qt, bh;
  if (CAUSAL) {
    // Heads in groups whose K/V fit in a share of L2, one group after the
    // other; within a group the longest units first (query blocks from the
    // end of the sequence), the group's heads fastest.  The CTAs working at
    // the same time then read the K/V of one group only.  (The last group
    // may hold fewer heads.)
    const int grp = p.fd_group_units.div(t);
    const int w = t - grp * p.head_group * p.n_qtiles;
    const FastDiv& fh = grp == p.last_group ? p.fd_last_heads : p.fd_group_heads;
    const int wq = fh.div(w);
    qt = p.n_qtiles - 1 - wq;
    bh = grp * p.head_group + (w - wq * static_cast<int>(fh.d));
  } else {       // consecutive units share a head, so its K/V stay hot in L2
    bh = p.fd_qtiles.div(t);
    qt = t - bh * p.n_qtiles;
  }
  u.b = p.fd_H.div(bh);
  u.h = bh - u.b * p.H;
  u.q0 = qt * kBQ;
  int kv, q_len;
  if (p.cu_q != nullptr) {
    // packed sequences: offsets clamped so that any content stays in bounds
    const int qs = min(max(__ldg(p.cu_q + u.b), 0), p.total_q);
    const int qe = min(max(__ldg(p.cu_q + u.b + 1), qs), p.total_q);
    q_len = qe - qs;
    u.q_tok0 = qs + u.q0;
    if (p.block_table != nullptr) {
      kv = min(max(__ldg(p.seqlens_k + u.b), 0), p.max_pages * p.page_size);
      u.k_tok0 = 0;
    } else {
      const int ks = min(max(__ldg(p.cu_k + u.b), 0), p.total_k);
      const int ke = min(max(__ldg(p.cu_k + u.b + 1), ks), p.total_k);
      kv = ke - ks;
      u.k_tok0 = ks;
    }
  } else {
    q_len = p.Sq;
    kv = p.Sk;
    if (p.kv_lens != nullptr) kv = min(max(__ldg(p.kv_lens + u.b), 0), p.Sk);
    u.q_tok0 = 0;
    u.k_tok0 = 0;
  }
  u.rows = max(min(kBQ, q_len - u.q0), 0);
  u.kv = kv;
  int lim = kv;
  if (CAUSAL) lim = min(lim, u.q0 + u.rows);  // last row of the tile + 1
  const int n_all = u.rows > 0 ? (lim + kBK - 1) / kBK : 0;
  u.j0 = p.fd_splits.div(u.split * n_all);
  u.n = p.fd_splits.div((u.split + 1) * n_all) - u.j0;
  return u;
}

// Row maximum of a thread's 64 raw scores (columns >= climit excluded when
// MASKED); 4 independent chains of three-input max.
template <bool MASKED>
__device__ __forceinline__ float half_row_max(const uint32_t (&s)[2][32], int climit) {
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int col = 0; col < 64; col += 2) {
    float x0 = u2f(s[col >> 5][col & 31]);
    float x1 = u2f(s[col >> 5][(col + 1) & 31]);
    if (MASKED) {
      x0 = (col < climit) ? x0 : -INFINITY;
      x1 = (col + 1 < climit) ? x1 : -INFINITY;
    }
    m4[(col >> 1) & 3] = max3(m4[(col >> 1) & 3], x0, x1);
  }
  return fmaxf(max3(m4[0], m4[1], m4[2]), m4[3]);
}

// p = 2^(s*c - mb) for a thread's 64 scores (one packed FMA per pair; masked
// columns give 0) into 32 bf16 pairs (FP8: 16 words of four E4M3 values, in
// pk[0..15]); returns the fp32 sum.  With WITH_MAX it also returns the maximum
// of the raw valid scores, found in the same pass.
template <bool MASKED, bool WITH_MAX, bool FP8 = false>
__device__ __forceinline__ float half_row_exp(const uint32_t (&s)[2][32], float c, float mb, int climit,
                                              uint32_t (&pk)[32], float& mx) {
  const uint64_t c2 = f2_pack(c, c);
  const uint64_t nmb2 = f2_pack(-mb, -mb);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  float pprev0 = 0.0f, pprev1 = 0.0f;  // FP8: the previous pair, packed with the next
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const int col = 2 * e;
    const float s0 = u2f(s[col >> 5][col & 31]);
    const float s1 = u2f(s[col >> 5][(col + 1) & 31]);
    float x0, x1;
    f2_unpack(f2_fma(f2_pack(s0, s1), c2, nmb2), x0, x1);
    float p0 = ex2_approx(x0);
    float p1 = ex2_approx(x1);
    if (MASKED) {
      const bool v0 = col < climit;
      const bool v1 = col + 1 < climit;
      p0 = v0 ? p0 : 0.0f;
      p1 = v1 ? p1 : 0.0f;
      if (WITH_MAX) m4[e & 3] = max3(m4[e & 3], v0 ? s0 : -INFINITY, v1 ? s1 : -INFINITY);
    } else if (WITH_MAX) {
      m4[e & 3] = max3(m4[e & 3], s0, s1);
    }
    acc[e & 3] = f2_add(acc[e & 3], f2_pack(p0, p1));
    if constexpr (FP8) {
      if (e & 1) pk[e >> 1] = pack_e4m3x4(pprev0, pprev1, p0, p1);
      pprev0 = p0;
      pprev1 = p1;
    } else {
      pk[e] = pack_bf16x2(p0, p1);
    }
  }
  if (WITH_MAX) mx = fmaxf(max3(m4[0], m4[1], m4[2]), m4[3]);
  const uint64_t a01 = f2_add(acc[0], acc[1]);
  const uint64_t a23 = f2_add(acc[2], acc[3]);
  float lo, hi;
  f2_unpack(f2_add(a01, a23), lo, hi);
  return lo + hi;
}

// A thread's half of its O row (D/2 fp32 columns in TMEM) *= alpha.
template <int D>
__device__ __forceinline__ void rescale_o_half(uint32_t tO, float alpha) {
  const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
  for (int q = 0; q < D / 64; ++q) {
    uint32_t o[32];
    tmem_ld_32x32b_x32(tO + q * 32, o);
    tmem_ld_wait_x32(o);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float lo, hi;
      f2_unpack(f2_mul(f2_pack(u2f(o[2 * e]), u2f(o[2 * e + 1])), a2), lo, hi);
      o[2 * e] = __float_as_uint(lo);
      o[2 * e + 1] = __float_as_uint(hi);
    }
    tmem_st_32x32b_x32(tO + q * 32, o);
  }
}

// SPLIT: K and V in rings of their own, each with its own producer warp
// (packed and paged batches); otherwise one ring of alternating K and V tiles
// (see Geo).
template <int D, bool CAUSAL, bool FP8, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const Params p) {
  using G = Geo<D, FP8, SPLIT>;
  using PR = Prec<FP8>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = smem_addr(smem_raw);
  uint8_t* base_ptr = smem_raw;
  Ctrl& ctl = *reinterpret_cast<Ctrl*>(base_ptr);
  Xchg& xch = *reinterpret_cast<Xchg*>(base_ptr + 1024);
  volatile int* abort_flag = &ctl.abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The layout leaves no slack for aligning the 128-byte swizzle atoms: a
  // block whose dynamic shared memory does not start 1024-byte aligned
  // (never seen) reports it and does nothing, before touching anything.
  if ((base & 1023u) != 0u) {
    if (threadIdx.x == 0) record_give_up(kSiteAlign);
    return;
  }

  const uint32_t bar_q_full = smem_addr(&ctl.q_full);
  const uint32_t bar_q_empty = smem_addr(&ctl.q_empty);
  const uint32_t bar_k_full0 = smem_addr(&ctl.k_full[0]);
  const uint32_t bar_v_full0 = smem_addr(&ctl.v_full[0]);
  const uint32_t bar_kv_empty0 = smem_addr(&ctl.kv_empty[0]);
  // barrier of buffer b = barrier of buffer 0 + 8 * b (consecutive uint64_t)
  const uint32_t bar_s_full0 = smem_addr(&ctl.s_full[0]);
  const uint32_t bar_s_free0 = smem_addr(&ctl.s_free[0]);  // bf16 protocol: the softmax has read S_b
  const uint32_t bar_p_full0 = smem_addr(&ctl.p_full[0]);
  const uint32_t bar_p_free0 = smem_addr(&ctl.p_free[0]);  // P V of the buffer's tile done: P_b (and S_b) free
  const uint32_t bar_o_full0 = smem_addr(&ctl.o_full[0]);
  const uint32_t bar_o_free0 = smem_addr(&ctl.o_free[0]);
  const uint32_t bar_uq_full0 = smem_addr(&ctl.uq_full[0]);
  const uint32_t bar_uq_empty0 = smem_addr(&ctl.uq_empty[0]);
  volatile int* unit_q = ctl.unit_q;

  if (warp == 0) {
    // the barriers are initialised by the 32 lanes of warp 0, a few each
    // (one thread initialising all of them serially took ~1500 cycles)
    if (lane < G::kSlots) {
      mbar_init(bar_k_full0 + 8 * lane, 1);
      mbar_init(bar_v_full0 + 8 * lane, 1);
      mbar_init(bar_kv_empty0 + 8 * lane, 1);  // K slots: QK issuer; V slots: PV issuer
    } else if (lane >= 16 && lane < 18) {
      const int b = lane - 16;
      mbar_init(bar_s_full0 + 8 * b, 1);
      mbar_init(bar_s_free0 + 8 * b, kSoftmaxWarps);
      mbar_init(bar_p_full0 + 8 * b, kSoftmaxWarps);
      mbar_init(bar_p_free0 + 8 * b, 1);
    } else if (lane >= 18 && lane < 20) {
      const int b = lane - 18;
      mbar_init(bar_o_full0 + 8 * b, 1);
      mbar_init(bar_o_free0 + 8 * b, kSoftmaxWarps);
      mbar_init(smem_addr(&ctl.drain[b]), 1);
    } else if (lane >= 20 && lane < 20 + kUnitQ) {
      const int k = lane - 20;
      mbar_init(bar_uq_full0 + 8 * k, 1);
      mbar_init(bar_uq_empty0 + 8 * k, kUnitQReaders + (SPLIT ? 1 : 0));
    } else if (lane == 31) {
      mbar_init(bar_q_full, 1);
      mbar_init(bar_q_empty, 1);
      mbar_init(smem_addr(&ctl.pv_issued), 1);
      ctl.abort_flag = 0;
    }
    fence_barrier_init();
  }
  if (warp == kWarpQK) {
    tmem_alloc(smem_addr(&ctl.tmem_base), G::kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  if (warp == kWarpLoad && lane == 0) {
    prefetch_tensor_map(&map_q);
    prefetch_tensor_map(&map_k);
    prefetch_tensor_map(&map_v);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = ctl.tmem_base;
  const uint64_t limit = p.wait_limit_ns;
  // every role walks the same sequence of units (whole rounds of gridDim.x)
  const int t_end = (p.total_units + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x) *
                    static_cast<int>(gridDim.x);

  // K/V tile layout (Geo): split rings (packed and paged batches) or one ring
  constexpr bool split = SPLIT;

  if (warp >= kSoftmaxWarps) {
    regs_decrease<kRegsOther>();
  // The two 64-key halves of tile j of unit u in a paged cache, as token rows
  // of the cache; a half past the sequence's keys is read from one row past
  // the cache: zeros.  (Both lookups are in flight together.)
  auto lookup_pages = [&](const Unit& u, int j, int (&page_tok)[2]) {
    page_tok[0] = page_tok[1] = p.cache_tokens;
    if (p.block_table == nullptr) return;
    const int key0 = (u.j0 + j) * kBK;
    int pg[2] = {0, 0};
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int pos = key0 + 64 * hf;
      if (pos < u.kv) pg[hf] = __ldg(p.block_table + static_cast<size_t>(u.b) * p.max_pages + pos / p.page_size);
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int pos = key0 + 64 * hf;
      if (pos < u.kv) page_tok[hf] = min(max(pg[hf], 0), p.num_pages - 1) * p.page_size + pos % p.page_size;
    }
  };
  // K_j (is_v false) or V_j of unit u into ring slot `slot`, completing on `full`
  auto load_tile = [&](bool is_v, uint32_t slot, uint32_t full, const Unit& u, int j, const int (&page_tok)[2],
                       uint64_t pol) {
    mbar_arrive_expect_tx(full, G::kTileBytes);
    const CUtensorMap* m = is_v ? &map_v : &map_k;
    const int key0 = (u.j0 + j) * kBK;
    const uint32_t dst = base + G::kOffRing + slot * G::kTileBytes;
    const bool packed = p.cu_q != nullptr;  // padded maps are (D, S, H, B); packed maps are (D, H, tokens, 1)
    if (FP8 && is_v && !p.v_rows) {
      // E4M3 V given transposed, (Sk, D, H, B): the tile is D rows, each 128
      // keys long (K-major for the P V product)
      tma_load_4d_hint(dst, m, full, key0, 0, u.h, u.b, pol);
    } else if (p.block_table == nullptr) {
      for (int c = 0; c < G::kChunks; ++c)
        tma_load_4d_hint(dst + c * G::kChunkBytes, m, full, c * G::kChunkElems, packed ? u.h : key0,
                         packed ? u.k_tok0 + key0 : u.h, packed ? 0 : u.b, pol);
    } else {
      // paged: two 64-key boxes, each inside one page (page_size is a
      // multiple of 64)
      for (int hf = 0; hf < 2; ++hf)
        for (int c = 0; c < G::kChunks; ++c)
          tma_load_4d_hint(dst + c * G::kChunkBytes + hf * (G::kChunkBytes / 2), m, full, c * 64, u.h,
                           page_tok[hf], 0, pol);
    }
  };
  // Drains of a producer lane before the CTA exits: after a failure, every
  // copy it started must land; in any case the issuers' last commit arrivals
  // on the empty barriers of its slots (nothing else waits for them) must
  // have landed before this CTA's shared memory is gone.
  auto drain_slots = [&](bool with_k, bool with_v, uint32_t k_issued, uint32_t v_issued, bool failed) {
    if constexpr (!SPLIT) {
      // one ring: positions 0 .. ring-1 were issued (K_t at 2t, V_t at 2t+1)
      const uint32_t ring = k_issued + v_issued;
      for (uint32_t s = 0; s < static_cast<uint32_t>(G::kSlots) && s < ring; ++s) {
        const uint32_t last = ring - 1 - ((ring - 1 - s) % G::kSlots);  // last position issued into slot s
        const typename G::Fill f = G::fill_of(last >> 1, (last & 1u) != 0, false);
        if (failed) wait_phase_drain(((last & 1u) ? bar_v_full0 : bar_k_full0) + 8 * s, f.full_use & 1u);
        wait_phase_drain(bar_kv_empty0 + 8 * s, f.empty_use & 1u);
      }
    } else {
      // split rings: ring r of n slots from slot `first` got `issued` fills in order
      for (int kind = 0; kind < 2; ++kind) {
        const bool is_v = kind == 1;
        if (is_v ? !with_v : !with_k) continue;
        const uint32_t issued = is_v ? v_issued : k_issued;
        const uint32_t first = is_v ? static_cast<uint32_t>(G::kSlotsK) : 0u;
        const uint32_t n = is_v ? static_cast<uint32_t>(G::kSlotsV) : static_cast<uint32_t>(G::kSlotsK);
        for (uint32_t i = 0; i < n && i < issued; ++i) {
          const uint32_t use = (issued - 1 - i) / n;  // phase index of the last fill of slot first + i
          if (failed) wait_phase_drain((is_v ? bar_v_full0 : bar_k_full0) + 8 * (first + i), use & 1u);
          wait_phase_drain(bar_kv_empty0 + 8 * (first + i), use & 1u);
        }
      }
    }
  };
  if (warp == kWarpLoad) {
    // ------------------------------------------- TMA: units, Q, K (and V)
    if (lane == 0) {
      const uint64_t pol_keep = l2_policy_evict_last();   // K/V: re-read by every query block of the head
      const uint64_t pol_once = l2_policy_evict_first();  // Q: read once
      uint32_t k_issued = 0, v_issued = 0, qcount = 0, kq = 0;
      int t_static = blockIdx.x;
      bool ok = true;
      while (ok) {
        // The next unit with rows: claimed from the launch's counter (dynamic:
        // any CTA takes the next unit in the units' own order, longest first
        // when causal) or dealt round-robin; pushed to the CTA's unit queue.
        int unit = -1;
        Unit u;
        for (;;) {
          int cand;
          if (p.sched != nullptr) {
            cand = static_cast<int>(atomicAdd(p.sched, 1u));
            if (cand >= p.total_units) break;
          } else {
            if (t_static >= t_end) break;
            cand = unit_at<CAUSAL>(p, t_static);
            t_static += gridDim.x;
            if (cand >= p.total_units) continue;
          }
          u = decode_unit<CAUSAL>(p, cand);
          if (u.rows > 0) {
            unit = cand;
            break;
          }
        }
        {
          const uint32_t slot = kq % kUnitQ;
          if (!wait_phase(bar_uq_empty0 + 8 * slot, ((kq / kUnitQ) & 1u) ^ 1u, abort_flag, kSiteUnitQ, limit)) {
            ok = false;
            break;
          }
          unit_q[slot] = unit;
          mbar_arrive(bar_uq_full0 + 8 * slot);
          ++kq;
        }
        if (unit < 0) break;
        if (u.n == 0) continue;
        if (!wait_phase(bar_q_empty, (qcount & 1u) ^ 1u, abort_flag, kSiteQEmpty, limit)) { ok = false; break; }
        mbar_arrive_expect_tx(bar_q_full, G::kTileBytes);
        const bool packed = p.cu_q != nullptr;
        for (int c = 0; c < G::kChunks; ++c)
          tma_load_4d_hint(base + G::kOffQ + c * G::kChunkBytes, &map_q, bar_q_full, c * G::kChunkElems,
                           packed ? u.h : u.q0, packed ? u.q_tok0 : u.h, packed ? 0 : u.b, pol_once);
        ++qcount;
        for (int j = 0; ok && j < u.n; ++j) {
          int page_tok[2];
          lookup_pages(u, j, page_tok);
          for (int sel = 0; sel < (split ? 1 : 2); ++sel) {  // K_j, then (single ring) V_j
            const typename G::Fill f = G::fill_of(sel ? v_issued : k_issued, sel != 0, split);
            if (!wait_phase(bar_kv_empty0 + 8 * f.slot, (f.empty_use & 1u) ^ 1u, abort_flag, kSiteKvEmpty, limit)) {
              ok = false;
              break;
            }
            if (!(sel == 0 && blockIdx.x == 0 && static_cast<int>(k_issued) == p.selftest_skip_fill))
              load_tile(sel != 0, f.slot, (sel ? bar_v_full0 : bar_k_full0) + 8 * f.slot, u, j, page_tok, pol_keep);
            if (sel) ++v_issued; else ++k_issued;
          }
        }
      }
      if (!ok && qcount > 0) wait_phase_drain(bar_q_full, (qcount - 1) & 1u);
      if (qcount > 0) wait_phase_drain(bar_q_empty, (qcount - 1) & 1u);
      drain_slots(true, !split, k_issued, v_issued, !ok);
      // Dynamic scheduling: this CTA makes no more claims.  The last CTA to get
      // here (every CTA does, aborting or not) puts the counter back to 0 for
      // the next launch that uses it.
      if (p.sched != nullptr) {
        __threadfence();
        if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
          atomicExch(p.sched, 0u);
          atomicExch(p.sched + 1, 0u);
        }
      }
    }
    __syncwarp();
  } else if (SPLIT && warp == kWarpLoadV) {
    // ----------------------------------------------------------- TMA: V
    // Split rings only: V tiles have a producer of their own, so that a V
    // fill waiting for its slot (free once that tile's P V completes) or for
    // its page lookup never holds up the K fills.  Units come from the CTA's
    // unit queue, of which this warp is then a reader.
    const uint64_t pol_keep = l2_policy_evict_last();
    uint32_t v_issued = 0, kq = 0;  // (lane 0)
    bool ok = true;
    while (ok) {
      const int unit = take_unit(kq, unit_q, bar_uq_full0, bar_uq_empty0, abort_flag, limit, lane);
      if (unit == -2) { ok = false; break; }
      if (unit < 0) break;
      const Unit u = decode_unit<CAUSAL>(p, unit);
      if (u.n == 0) continue;
      if (lane == 0) {
        for (int j = 0; j < u.n; ++j) {
          int page_tok[2];
          lookup_pages(u, j, page_tok);
          const typename G::Fill f = G::fill_of(v_issued, true, true);
          if (!wait_phase(bar_kv_empty0 + 8 * f.slot, (f.empty_use & 1u) ^ 1u, abort_flag, kSiteKvEmpty, limit)) {
            ok = false;
            break;
          }
          load_tile(true, f.slot, bar_v_full0 + 8 * f.slot, u, j, page_tok, pol_keep);
          ++v_issued;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0) drain_slots(false, true, 0, v_issued, !ok);
    __syncwarp();
  } else if (warp == kWarpQK) {
    // ---------------------------------------------------- S = Q K^T issuer
    // Runs up to two tiles ahead of the softmax (two S buffers).  Releases
    // each K slot once its MMAs complete.
    uint32_t qcount = 0, tcount = 0, kq = 0;
    bool ok = true;
    const uint32_t qa = base + G::kOffQ;
    const uint32_t bar_pv_issued = smem_addr(&ctl.pv_issued);
    while (ok) {
      const int unit = take_unit(kq, unit_q, bar_uq_full0, bar_uq_empty0, abort_flag, limit, lane);
      if (unit == -2) { ok = false; break; }
      if (unit < 0) break;
      const Unit u = decode_unit<CAUSAL>(p, unit);
      if (u.n == 0) continue;
      if (!wait_warp(bar_q_full, qcount & 1u, abort_flag, kSiteQFull, limit)) { ok = false; break; }
      // The unit's first S = Q K^T goes into the tensor pipe after the last
      // P V of the unit before: queued ahead of it, the products of this unit
      // would delay that unit's O (and the epilogue of the softmax warps, who
      // need this S only after it) by two QK^T products.
      if (qcount > 0 && !wait_warp(bar_pv_issued, (qcount - 1) & 1u, abort_flag, kSitePvIssued, limit)) {
        ok = false;
        break;
      }
      ++qcount;
      for (int j = 0; j < u.n; ++j, ++tcount) {
        const uint32_t b = tcount & 1u;
        const uint32_t use = tcount >> 1;
        if (tcount >= 2) {
          // S_b is free once the softmax has read S of tile tcount-2 (bf16), or
          // once the P V of tile tcount-2 has consumed the P written over it
          const uint32_t bar_sb = (G::kPInS ? bar_p_free0 : bar_s_free0) + 8 * b;
          if (!wait_warp(bar_sb, (use - 1) & 1u, abort_flag, kSiteSFree, limit)) { ok = false; break; }
          tc_fence_after_sync();
        }
        const typename G::Fill f = G::fill_of(tcount, false, split);
        const uint32_t slot = f.slot;
        if (!wait_warp(bar_k_full0 + 8 * slot, f.full_use & 1u, abort_flag, kSiteKvFull, limit)) {
          ok = false;
          break;
        }
        // S_b = Q K_j^T: both operands K-major, 128-B swizzled; one MMA per 16 columns of D.
        const uint32_t ka = base + G::kOffRing + slot * G::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < G::kKSteps; ++kk) {
          const uint32_t off = (kk >> 2) * G::kChunkBytes + (kk & 3) * 32;
          if constexpr (FP8)
            mma_ss_f8_elect(tmem + G::kTmemS + 128u * b, sdesc_sw(qa + off, 16, G::kSbo, G::kSwMode),
                            sdesc_sw(ka + off, 16, G::kSbo, G::kSwMode), p.idesc_qk, kk > 0 ? 1u : 0u);
          else
            mma_ss_elect(tmem + G::kTmemS + 128u * b, sdesc_sw(qa + off, 16, G::kSbo, G::kSwMode),
                         sdesc_sw(ka + off, 16, G::kSbo, G::kSwMode), p.idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit_elect(bar_s_full0 + 8 * b);
        mma_commit_elect(bar_kv_empty0 + 8 * slot);
      }
      if (!ok) break;
      mma_commit_elect(bar_q_empty);
    }
    if (!ok) {
      const uint32_t bar_d = smem_addr(&ctl.drain[0]);
      mma_commit_elect(bar_d);
      wait_phase_drain(bar_d, 0);
    }
  } else if (warp == kWarpPV) {
    // ---------------------------------------------------- O += P V issuer
    // Consecutive units alternate between the two O buffers, so a unit's
    // products never wait for the epilogue of the unit before.
    uint32_t tcount = 0, ucount = 0, kq = 0;
    bool ok = true;
    while (ok) {
      const int unit = take_unit(kq, unit_q, bar_uq_full0, bar_uq_empty0, abort_flag, limit, lane);
      if (unit == -2) { ok = false; break; }
      if (unit < 0) break;
      const Unit u = decode_unit<CAUSAL>(p, unit);
      if (u.n == 0) continue;
      for (int j = 0; j < u.n; ++j, ++tcount) {
        const uint32_t b = tcount & 1u;
        const uint32_t use = tcount >> 1;
        if (!wait_warp(bar_p_full0 + 8 * b, use & 1u, abort_flag, kSitePFull, limit)) { ok = false; break; }
        const uint32_t ob = ucount % G::kOBufs;
        if (G::kPInS && j == 0 && ucount >= 2 &&  // the epilogue two units back has read O buffer ob
            !wait_warp(bar_o_free0 + 8 * ob, ((ucount >> 1) - 1) & 1u, abort_flag, kSiteOFull, limit)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t tOb = tmem + G::kTmemO + static_cast<uint32_t>(D) * ob;
        // the tile's P: over its S buffer, or in its own P buffer
        const uint32_t tSb = tmem + (G::kPInS ? G::kTmemS + 128u * b : G::kTmemP + 64u * b);
        const typename G::Fill f = G::fill_of(tcount, true, split);
        const uint32_t slot = f.slot;
        if (!wait_warp(bar_v_full0 + 8 * slot, f.full_use & 1u, abort_flag, kSiteKvFull, limit)) {
          ok = false;
          break;
        }
        const uint32_t va = base + G::kOffRing + slot * G::kTileBytes;
        if constexpr (FP8) {
          // O += P_b V_j with E4M3 P (32 keys = 8 columns per MMA, four per
          // column).  V given transposed: K-major in shared memory (D rows of
          // 128 keys, 128-byte swizzle), 32 keys = 32 bytes along each row per
          // MMA.  V in rows: MN-major (rows of keys, D contiguous: one swizzle
          // atom wide, 128 or 64 bytes), 32 keys = 32 rows per MMA.
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk) {
            const uint64_t vdesc =
                p.v_rows ? sdesc_sw(va + kk * 32 * G::kRowBytes, 16, G::kSbo, G::kSwMode)
                         : sdesc_sw(va + kk * 32, 16, 1024, kSmemSwizzle128B);
            mma_ts_f8_elect(tOb, tSb + G::p_col(kk), vdesc, p.idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
          }
        } else {
          // O += P_b V_j: P from TMEM (16 keys = 8 columns per MMA), V MN-major in
          // smem (LBO = distance between 64-column chunks of D, SBO = 8 keys x 128 B).
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            mma_ts_elect(tOb, tSb + G::p_col(kk), sdesc_sw128(va + kk * 16 * 128, G::kChunkBytes, 1024),
                         p.idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit_elect(bar_p_free0 + 8 * b);
        mma_commit_elect(bar_kv_empty0 + 8 * slot);
        if (j == u.n - 1) {
          mma_commit_elect(bar_o_full0 + 8 * ob);
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&ctl.pv_issued));  // the next unit's first QK^T may follow
        }
      }
      if (!ok) break;
      ++ucount;
    }
    if (!ok) {
      const uint32_t bar_d = smem_addr(&ctl.drain[1]);
      mma_commit_elect(bar_d);
      wait_phase_drain(bar_d, 0);
    }
  }
  } else {
    regs_increase<kRegsSoftmax>();
    // -------------------------------------------------------------- softmax
    // Two threads per query row: half 0 (warps 0-3) owns columns 0-63 of each
    // score tile, half 1 (warps 4-7) columns 64-127.  Both keep the same
    // reference max (when a row may have grown they exchange their partial
    // maxima through shared memory and the pair's named barrier) and their
    // own partial row sums, added in the epilogue.
    //
    // The two halves of a row are warps w and w + 4; each such pair has its own
    // named barrier (id 1 + w, 64 threads), so pairs never wait on each other.
    // Named barriers cannot time out, so the pair keeps one discipline: a wait
    // that fails only marks the warp as failed and skips work; both warps
    // execute every barrier of the pair; and every decision to leave is the OR
    // of the abort flag over the pair, reduced by the barrier itself, so both
    // warps take it together.
    const int half = warp >> 2;
    const int r = threadIdx.x & (kBQ - 1);         // row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c = p.c;
    const uint32_t bar_pair = 1u + static_cast<uint32_t>(warp & 3);
    constexpr uint32_t kPairThreads = 64;
    uint32_t tcount = 0, ocount = 0, kq = 0;
    bool ok = true;

    // The next unit is taken from the queue before a unit's epilogue, under
    // the wait for the unit's last P V (pend != -3).
    int pend = -3;
    while (ok) {
      int unit = pend;
      if (pend != -3) {
        pend = -3;
      } else {
        unit = take_unit(kq, unit_q, bar_uq_full0, bar_uq_empty0, abort_flag, limit, lane);
        // both warps of the pair read the same entry; they leave together if
        // either gave up or the CTA aborts
        if (named_bar_red_or(bar_pair, kPairThreads, unit == -2 || *abort_flag != 0)) { ok = false; break; }
      }
      if (unit < 0) break;
      const Unit u = decode_unit<CAUSAL>(p, unit);
      const int row = u.q0 + r;     // position of this thread's query row within its sequence
      const bool row_ok = r < u.rows;
      size_t row_index, lse_index;  // row of O (in units of D elements) and index into lse
      if (p.cu_q != nullptr) {      // packed: o [total_q, H, D], lse [H, total_q]
        const size_t tok = static_cast<size_t>(u.q_tok0) + r;
        row_index = tok * p.H + u.h;
        lse_index = static_cast<size_t>(u.h) * p.total_q + tok;
      } else {                      // padded: o [B, H, Sq, D], lse [B, H, Sq]
        row_index = (static_cast<size_t>(u.b) * p.H + u.h) * static_cast<size_t>(p.Sq) + row;
        lse_index = row_index;
      }
      uint16_t* o_dst = p.o + row_index * D + (D / 2) * half;
      // split mode (padded only): this key range's partial row
      const size_t prow = static_cast<size_t>(u.split) * p.B * p.H * static_cast<size_t>(p.Sq) + row_index;
      float* op_dst = (p.o_part != nullptr) ? p.o_part + prow * D + (D / 2) * half : nullptr;
      if (u.n == 0) {  // no valid key for any row of this unit: O = 0, LSE = -inf
        if (row_ok) {
          if (op_dst == nullptr) {
            uint4* dst = reinterpret_cast<uint4*>(o_dst);
#pragma unroll
            for (int q = 0; q < D / 16; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
            if (half == 0) p.lse[lse_index] = -INFINITY;
          } else {
            float4* dst = reinterpret_cast<float4*>(op_dst);
#pragma unroll
            for (int q = 0; q < D / 8; ++q) dst[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (half == 0) p.lse_part[prow] = -INFINITY;
          }
        }
        continue;
      }

      // this unit's O buffer (units with keys alternate, as in the P V issuer)
      const uint32_t ob = ocount % G::kOBufs;
      const uint32_t tO = tmem + lane_off + G::kTmemO + static_cast<uint32_t>(D) * ob + (D / 2) * half;
      float m_used = -INFINITY;  // reference max (log2 units, scale folded in), shared by both halves
      float l = 0.0f;            // this half's sum of 2^(x - m_used)
      bool failed = false;
      for (int j = 0; j < u.n; ++j, ++tcount) {
        const uint32_t b = tcount & 1u;
        const uint32_t use = tcount >> 1;
        const int k0 = (u.j0 + j) * kBK;
        const bool masked = (k0 + kBK > u.kv) || (CAUSAL && k0 + kBK - 1 > u.q0);
        int climit = u.kv - k0;  // columns >= climit of the tile are masked for this row
        if (CAUSAL) climit = min(climit, row - k0 + 1);
        climit -= 64 * half;     // ... in this half's column numbering

        uint32_t s[2][32];
        uint32_t pk[32];
        float sum = 0.0f;
        bool pf_ready = true;
        bool suspect = false;  // this thread's part of the row may have grown past the reference
        if (!failed && !wait_warp(bar_s_full0 + 8 * b, use & 1u, abort_flag, kSiteSFull, limit)) failed = true;
        if (!failed) {
          tc_fence_after_sync();
          const uint32_t tS = tmem + lane_off + G::kTmemS + 128u * b + 64u * half;
          tmem_ld_32x32b_x32(tS, s[0]);
          tmem_ld_32x32b_x32(tS + 32, s[1]);
          tmem_ld_wait_x32(s[0]);
          tmem_ld_wait_x32(s[1]);
          if constexpr (!G::kPInS) {
            warp_arrive_after_tc(bar_s_free0 + 8 * b, lane);  // the QK issuer may refill S_b
            // P buffer b is free once the P V of tile tcount-2 has completed:
            // ask now, use the answer after the exponentials.
            if (tcount >= 2) pf_ready = mbar_test_wait(bar_p_free0 + 8 * b, (use - 1) & 1u);
          }
          // (P over S: P_b goes over the columns just read; S_b was written
          // after the P V of tile tcount-2 had consumed the previous P_b.)
          if (j > 0) {
            // Exponentiate against the current reference right away.  Each term
            // is 2^(x - m_used + shift); if they all stay <= 2^(tau + shift) no
            // score of this part of the row grew past the reference by more than
            // tau, and a part sum <= 2^(tau + shift) proves it (the test is also
            // false for NaN / inf).
            float unused;
            sum = masked ? half_row_exp<true, false, FP8>(s, c, m_used - PR::kShift, climit, pk, unused)
                         : half_row_exp<false, false, FP8>(s, c, m_used - PR::kShift, climit, pk, unused);
            suspect = !(sum <= PR::kSumLimit);
          } else {
            suspect = true;  // first tile: the reference is this tile's row max
          }
        }
        // One barrier per tile for the pair; it also tells both warps whether
        // any of their rows needs its exact maximum (or the CTA is aborting).
        const bool any_suspect = named_bar_red_or(bar_pair, kPairThreads, suspect || *abort_flag != 0);
        bool rescale = false;
        float alpha = 1.0f;
        if (any_suspect) {
          // Exact row max: partial maxima of both halves through shared memory
          // (by tile parity, so a slow partner still reads the previous value
          // undisturbed).  The second barrier publishes them and settles abort.
          if (!failed) {
            xch.xmax[b][half][r] = masked ? half_row_max<true>(s, climit) : half_row_max<false>(s, climit);
          }
          if (named_bar_red_or(bar_pair, kPairThreads, *abort_flag != 0)) { ok = false; break; }
          const float mx = fmaxf(xch.xmax[b][0][r], xch.xmax[b][1][r]);
          const float m_tile = (mx == -INFINITY) ? -INFINITY : mx * c;
          if (j == 0) {
            // First tile: its row max is the reference (every row of a unit with
            // n > 0 has key 0 valid, so the reference is finite afterwards).
            m_used = m_tile;
            const float mb = (m_used == -INFINITY) ? 0.0f : m_used - PR::kShift;
            float unused;
            sum = masked ? half_row_exp<true, false, FP8>(s, c, mb, climit, pk, unused)
                         : half_row_exp<false, false, FP8>(s, c, mb, climit, pk, unused);
          } else {
            // Lazy correction: only when the max grew by more than tau is the
            // reference moved, this tile recomputed, and l and O rescaled by
            // alpha = 2^(m_old - m_new); every term stays <= 2^(tau + shift) and O and l
            // always share one reference.  Both halves see the same row max, so
            // they take the same decision.
            const bool grow = m_tile > m_used + PR::kTau;
            if (__any_sync(0xffffffffu, grow)) {
              rescale = true;
              if (grow) {
                alpha = ex2_approx(m_used - m_tile);
                m_used = m_tile;
              }
              float unused;
              sum = masked ? half_row_exp<true, false, FP8>(s, c, m_used - PR::kShift, climit, pk, unused)
                           : half_row_exp<false, false, FP8>(s, c, m_used - PR::kShift, climit, pk, unused);
            }
          }
        }
        if (!G::kPInS && !pf_ready &&
            !wait_warp(bar_p_free0 + 8 * b, (use - 1) & 1u, abort_flag, kSitePFree, limit))
          failed = true;
        if (rescale && !failed) {
          // O is stable once the PV of the previous tile (buffer b^1) completed.
          const uint32_t tp = tcount - 1;
          if (!wait_warp(bar_p_free0 + 8 * (tp & 1u), (tp >> 1) & 1u, abort_flag, kSitePFree, limit)) {
            failed = true;
          } else {
            tc_fence_after_sync();
            l *= alpha;
            rescale_o_half<D>(tO, alpha);
          }
        }
        if (!failed) {
          tc_fence_after_sync();
          const uint32_t tP = tmem + lane_off +
                              (G::kPInS ? G::kTmemS + 128u * b + 64u * half    // over this half's S
                                        : G::kTmemP + 64u * b + 32u * half);   // own P buffer
          if constexpr (FP8) {  // 64 keys x 1 B = 16 columns
            tmem_st_32x32b_x16(tP, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
          } else {              // 64 keys x 2 B = 32 columns
            tmem_st_32x32b_x16(tP, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
            tmem_st_32x32b_x16(tP + 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]));
          }
          tmem_st_wait();
          warp_arrive_after_tc(bar_p_full0 + 8 * b, lane);
          l += sum;
        }
      }
      if (!ok) break;

      // the next unit (see above); the pair leaves together on a failure
      pend = take_unit(kq, unit_q, bar_uq_full0, bar_uq_empty0, abort_flag, limit, lane);
      if (named_bar_red_or(bar_pair, kPairThreads, pend == -2 || *abort_flag != 0)) { ok = false; break; }

      // ------------------------------------------------------------ epilogue
      if (!failed &&
          !wait_warp(bar_o_full0 + 8 * ob, (ocount / G::kOBufs) & 1u, abort_flag, kSiteOFull, limit))
        failed = true;
      ++ocount;
      const uint32_t bsum = ((tcount - 1u) & 1u) ^ 1u;  // the parity the unit's last tile did not use
      if (!failed) xch.xmax[bsum][half][r] = l;
      if (named_bar_red_or(bar_pair, kPairThreads, *abort_flag != 0)) { ok = false; break; }
      tc_fence_after_sync();
      const float l_row = l + xch.xmax[bsum][half ^ 1][r];
      const bool has_key = l_row > 0.0f;
      // hardware reciprocal and log2 (relative errors near 2^-23; O is
      // rounded to bf16, LSE is compared at 1e-3)
      const float inv_l = has_key ? p.v_scale * rcp_approx(l_row) : 0.0f;
      const float lse_row = has_key ? (m_used - PR::kShift + lg2_approx(l_row)) * kLn2 : -INFINITY;
#pragma unroll
      for (int q = 0; q < D / 64; ++q) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tO + q * 32, o);
        tmem_ld_wait_x32(o);
        if (row_ok) {
          if (op_dst == nullptr) {
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              w[e] = has_key ? pack_bf16x2(u2f(o[2 * e]) * inv_l, u2f(o[2 * e + 1]) * inv_l) : 0u;
            // The warp's 32 threads write 32 different rows, so each store
            // instruction touches 32 lines: 32-byte stores (when O is 32-byte
            // aligned, as every row half then is) halve the instructions and
            // write whole sectors.
            if (p.o_align32) {
              st_global_v8(o_dst + q * 32, *reinterpret_cast<const uint32_t(*)[8]>(&w[0]));
              st_global_v8(o_dst + q * 32 + 16, *reinterpret_cast<const uint32_t(*)[8]>(&w[8]));
            } else {
              uint4* dst = reinterpret_cast<uint4*>(o_dst + q * 32);
#pragma unroll
              for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
            }
          } else {  // normalised fp32 partial output (the workspace is 256-byte aligned)
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = has_key ? __float_as_uint(u2f(o[e]) * inv_l) : 0u;
#pragma unroll
            for (int e = 0; e < 4; ++e)
              st_global_v8(op_dst + q * 32 + 8 * e, *reinterpret_cast<const uint32_t(*)[8]>(&o[8 * e]));
          }
        }
      }
      if constexpr (G::kPInS) {
        // O buffer ob has been read: the unit two units later may use it
        warp_arrive_after_tc(bar_o_free0 + 8 * ob, lane);
      } else {
        // one O buffer: the next unit's first P V overwrites it only after every
        // softmax warp has arrived on p_full for it, which comes after this
        tc_fence_before_sync();
      }
      if (row_ok && half == 0) {
        if (op_dst == nullptr) p.lse[lse_index] = lse_row;
        else p.lse_part[prow] = lse_row;
      }
    }
    // The last p_free arrivals (commits of the last two PVs) land
    // asynchronously and nothing else waits for them: wait before exiting.
    for (uint32_t back = 1; back <= 2 && back <= tcount; ++back) {
      const uint32_t tp = tcount - back;
      wait_phase_drain(bar_p_free0 + 8 * (tp & 1u), (tp >> 1) & 1u);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpQK) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, G::kTmemCols);
  }
}

__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nothing ever arrives on `bar`: the bounded wait must give up.
    (void)wait_phase(smem_addr(&bar), 0, &abort_flag, kSiteSelftest, limit_ns);
  }
  __syncthreads();
}

// The forward kernel's launch shape with none of its work (mode 0), or with
// only its fixed per-block set-up and tear-down (mode 1): mbarrier
// initialisation, the 512-column Tensor Memory allocation, the block-wide
// synchronisations and the release.  The host requires one block per SM
// (the forward's shared memory), so allocations never wait on each other.
__global__ void __launch_bounds__(kThreads, 1) launch_floor_kernel(int mode) {
  if (mode == 0) return;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  Ctrl& ctl = *reinterpret_cast<Ctrl*>(smem_raw + (base - raw));
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < 12; ++s) mbar_init(smem_addr(&ctl.k_full[s]), 1);
    fence_barrier_init();
  }
  if (warp == kWarpQK) {
    tmem_alloc(smem_addr(&ctl.tmem_base), 512);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = ctl.tmem_base;
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpQK) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------- host side

struct DeviceInfo {
  int initialised = 0;
  int supported = 0;
  int num_sms = 0;
  // dynamic shared memory attribute set for kernel instantiation i (set at
  // most once; two host threads may both set it, which is harmless)
  std::atomic<bool> smem_set[14] = {};
  std::atomic<bool> bwd_smem_set[4] = {};
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

attn_status device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.initialised) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    d.num_sms = sms;
    d.initialised = 1;
  }
  if (!d.supported) return ATTN_ERR_UNSUPPORTED_DEVICE;
  *out = &d;
  return ATTN_OK;
}

// The tensor-map encoder is a driver function; it is fetched through the
// runtime so that the library itself does not link against libcuda (it then
// loads on machines without a driver, where every call reports ATTN_ERR_CUDA).
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// Rank-4 map over [B, H, S, D] (D innermost) with a 64 x box_rows box (one
// 128-B swizzle column of a tile).  Rows past S read as zeros and never spill
// into the next head.
bool make_map(CUtensorMap* m, const void* ptr, int B, int H, int S, int D, int box_rows = 128) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = encoder();
  if (encode == nullptr) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)S * D * 2, (cuuint64_t)H * S * D * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rank-4 maps over E4M3 tensors (one byte per element), (inner, rows, H, B)
// with a box of box_inner bytes x box_rows rows, swizzled to the box's row
// length (128 or 64 bytes).  Q, K and V in rows [B,H,S,D] as (D, S, H, B),
// boxes of 128 rows of D bytes; V^T [B,H,D,Sk] as (Sk, D, H, B), boxes of D
// rows, each 128 keys long.  Bytes past an edge read as zeros.
bool make_map_e4m3(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, int H, int B, uint32_t box_inner,
                   uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = encoder();
  if (encode == nullptr) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)inner, (cuuint64_t)(inner * rows), (cuuint64_t)(inner * rows * H)};
  const cuuint32_t box[4] = {box_inner, box_rows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle sw = box_inner == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rank-4 map over a packed [tokens, H, D] tensor as (D, H, tokens, 1) with a
// 64 x 1 x box_rows box: a 128-row box lands in shared memory as the same
// 128 rows x 128 B tile as the padded map's, a 64-row box as its upper or lower
// half.  Token rows past the end read as zeros.
bool make_map_packed(CUtensorMap* m, const void* ptr, int H, int total, int D, int box_rows = 128) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = encoder();
  if (encode == nullptr) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)total, 1};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)total * H * D * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Heads per causal group: as many as keep their K and V within 48 MB of L2
// (K/V bytes of one head = 2 * keys * D * element size).  Each group's units
// come longest first, so a last group of less than half the others' size
// would put its long units at the end of the launch; then the heads are
// spread evenly over the same number of groups (measured, causal D = 128:
// 32 heads at 4096 keys, 24 + 8 heads 968 TFLOP/s, 16 + 16 heads 1077; 64
// heads at 8192 keys 1352 against 1401; evening out groups that were already
// at least half full cost up to 5 %, so those stay as they are).
int head_group_for(int bh_count, int keys, int D, int elem_bytes) {
  const uint64_t bh = static_cast<uint64_t>(bh_count > 0 ? bh_count : 1);
  const uint64_t per_head = 2ull * static_cast<uint64_t>(keys > 0 ? keys : 1) * D * elem_bytes;
  uint64_t g = (48ull << 20) / per_head;
  if (g < 1) g = 1;
  if (g > bh) g = bh;
  const uint64_t groups = (bh + g - 1) / g;
  const uint64_t last = bh - (groups - 1) * g;
  if (groups > 1 && 2 * last < g) g = (bh + groups - 1) / groups;
  return static_cast<int>(g);
}

void clear_paged(Params& p) {
  p.block_table = nullptr;
  p.seqlens_k = nullptr;
  p.page_size = 0;
  p.max_pages = 0;
  p.num_pages = 0;
  p.cache_tokens = 0;
}

template <int D, bool CAUSAL, bool FP8 = false, bool SPLIT = false>
attn_status launch(DeviceInfo& dev, int idx, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                   const Params& p, cudaStream_t stream) {
  auto kern = attn_fwd_kernel<D, CAUSAL, FP8, SPLIT>;
  constexpr int smem = Geo<D, FP8, SPLIT>::kSmemBytes;
  if (!dev.smem_set[idx].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return ATTN_ERR_CUDA;
    dev.smem_set[idx].store(true, std::memory_order_release);
  }
  const int grid = p.total_units < dev.num_sms ? p.total_units : dev.num_sms;
  kern<<<grid, kThreads, smem, stream>>>(mq, mk, mv, with_divisors(p, grid));
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// LSE merge of key-range partial results: one warp per row, each lane owns
// D/32 consecutive columns.  M = max_s LSE_s, w_s = 2^((LSE_s - M) log2 e),
// O = sum_s w_s O_s / sum_s w_s, LSE = M + ln sum_s w_s; all-empty rows give
// O = 0 and LSE = -inf.
template <int D>
__global__ void __launch_bounds__(256) lse_merge_kernel(const float* __restrict__ o_parts,
                                                        const float* __restrict__ lse_parts, int n_parts,
                                                        long long rows, uint16_t* __restrict__ o,
                                                        float* __restrict__ lse) {
  constexpr int C = D / 32;
  constexpr float kLog2e = 1.4426950408889634f;
  const int lane = threadIdx.x & 31;
  const long long warp_id = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long n_warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long r = warp_id; r < rows; r += n_warps) {
    float m = -INFINITY;
    for (int s = 0; s < n_parts; ++s) m = fmaxf(m, __ldg(lse_parts + s * rows + r));
    float acc[C];
#pragma unroll
    for (int e = 0; e < C; ++e) acc[e] = 0.0f;
    float total = 0.0f;
    if (m != -INFINITY) {
      for (int s = 0; s < n_parts; ++s) {
        const float ls = __ldg(lse_parts + s * rows + r);
        if (ls == -INFINITY) continue;
        const float w = ex2_approx((ls - m) * kLog2e);
        total += w;
        const float* src = o_parts + (s * rows + r) * D + lane * C;
        if constexpr (C == 4) {
          const float4 x = __ldg(reinterpret_cast<const float4*>(src));
          acc[0] = fmaf(w, x.x, acc[0]);
          acc[1] = fmaf(w, x.y, acc[1]);
          acc[2] = fmaf(w, x.z, acc[2]);
          acc[3] = fmaf(w, x.w, acc[3]);
        } else {
          const float2 x = __ldg(reinterpret_cast<const float2*>(src));
          acc[0] = fmaf(w, x.x, acc[0]);
          acc[1] = fmaf(w, x.y, acc[1]);
        }
      }
    }
    const float inv = total > 0.0f ? 1.0f / total : 0.0f;
    uint16_t* dst = o + r * D + lane * C;
    if constexpr (C == 4) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                                  pack_bf16x2(acc[2] * inv, acc[3] * inv));
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
    if (lane == 0) lse[r] = total > 0.0f ? m + logf(total) : -INFINITY;
  }
}

attn_status launch_merge(DeviceInfo& dev, const float* o_parts, const float* lse_parts, int n_parts, long long rows,
                         int D, void* o, float* lse, cudaStream_t s) {
  if (rows == 0) return ATTN_OK;
  const long long warps_needed = rows;
  long long blocks = (warps_needed + 7) / 8;  // 8 warps per block
  const long long max_blocks = static_cast<long long>(dev.num_sms) * 8;
  if (blocks > max_blocks) blocks = max_blocks;
  if (D == 64)
    lse_merge_kernel<64><<<static_cast<int>(blocks), 256, 0, s>>>(o_parts, lse_parts, n_parts, rows,
                                                                   static_cast<uint16_t*>(o), lse);
  else
    lse_merge_kernel<128><<<static_cast<int>(blocks), 256, 0, s>>>(o_parts, lse_parts, n_parts, rows,
                                                                    static_cast<uint16_t*>(o), lse);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

constexpr int kMaxSplits = 128;

size_t round_up_256(size_t x) { return (x + 255) / 256 * 256; }

// Bytes of the split-mode workspace: partial O (fp32) then partial LSE (fp32).
size_t splitkv_bytes(int B, int H, int Sq, int D, int num_splits, size_t* lse_offset) {
  const size_t rows = static_cast<size_t>(B) * H * Sq;
  const size_t o_bytes = round_up_256(static_cast<size_t>(num_splits) * rows * D * sizeof(float));
  if (lse_offset != nullptr) *lse_offset = o_bytes;
  return o_bytes + round_up_256(static_cast<size_t>(num_splits) * rows * sizeof(float));
}

attn_status check_args(const void* q, const void* k, const void* v, const void* o, const float* lse, int B, int H,
                       int Sq, int Sk, int D, float scale, const int32_t* kv_lens, int num_splits) {
  if (B < 0 || H < 0 || Sq < 0 || Sk < 0) return ATTN_ERR_SHAPE;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED_D;
  if (!std::isfinite(scale)) return ATTN_ERR_SCALE;
  if (num_splits < 1 || num_splits > kMaxSplits) return ATTN_ERR_SHAPE;
  if (B == 0 || H == 0 || Sq == 0) return ATTN_OK;
  if (q == nullptr || o == nullptr || lse == nullptr) return ATTN_ERR_NULLPTR;
  if (Sk > 0 && (k == nullptr || v == nullptr)) return ATTN_ERR_NULLPTR;
  if (!aligned(q, 16) || !aligned(o, 16) || !aligned(lse, 4)) return ATTN_ERR_ALIGN;
  if (Sk > 0 && (!aligned(k, 16) || !aligned(v, 16))) return ATTN_ERR_ALIGN;
  if (kv_lens != nullptr && !aligned(kv_lens, 4)) return ATTN_ERR_ALIGN;
  // TMA strides must stay below 2^40 bytes; work units (whole rounds of the
  // persistent loop included) must fit an int.
  const uint64_t max_s = static_cast<uint64_t>(Sq > Sk ? Sq : Sk);
  if (static_cast<uint64_t>(H) * max_s * D * 2 >= (1ull << 40)) return ATTN_ERR_SHAPE;
  const uint64_t n_qtiles = (static_cast<uint64_t>(Sq) + kBQ - 1) / kBQ;
  if (static_cast<uint64_t>(B) * H * n_qtiles * num_splits > 0x7fff0000ull) return ATTN_ERR_SHAPE;
  return ATTN_OK;
}

// Launches the attention kernel.  o_part == nullptr: final bf16 O and LSE;
// otherwise num_splits key ranges write fp32 partials to o_part / lse_part.
// Parameters of a packed-query launch (variable-length or paged); the caller
// fills in the key side.
Params packed_params(void* o, float* lse, const int32_t* cu_q, int batch, int max_seqlen_q, int total_q, int H,
                     int D, float scale) {
  Params p;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.kv_lens = nullptr;
  p.B = batch;
  p.H = H;
  p.Sq = max_seqlen_q;
  p.Sk = 0;
  p.n_qtiles = static_cast<int>((static_cast<int64_t>(max_seqlen_q) + kBQ - 1) / kBQ);
  p.head_group = head_group_for(batch * H, max_seqlen_q, D, 2);  // sequence lengths are not known here
  p.num_splits = 1;
  p.total_units = static_cast<int>(static_cast<int64_t>(batch) * H * p.n_qtiles);  // checked by the caller
  p.o_part = nullptr;
  p.lse_part = nullptr;
  p.cu_q = cu_q;
  p.cu_k = nullptr;
  p.total_q = total_q;
  p.total_k = 0;
  clear_paged(p);
  p.sched = nullptr;
  p.c = static_cast<float>(std::fabs(static_cast<double>(scale)) * 1.4426950408889634);
  p.v_scale = 1.0f;
  p.idesc_qk = idesc_bf16_f32(kBQ, kBK, scale < 0.0f, false);
  p.idesc_pv = idesc_bf16_f32(kBQ, D, false, true);
  p.wait_limit_ns = kWaitLimitNs;
  return p;
}

// Packed and paged batches: the kernels with split K/V rings.
attn_status launch_any(DeviceInfo& dev, int D, bool causal, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, const Params& p, cudaStream_t s) {
  if (D == 64)
    return causal ? launch<64, true, false, true>(dev, 6, mq, mk, mv, p, s)
                  : launch<64, false, false, true>(dev, 7, mq, mk, mv, p, s);
  return causal ? launch<128, true, false, true>(dev, 8, mq, mk, mv, p, s)
                : launch<128, false, false, true>(dev, 9, mq, mk, mv, p, s);
}

attn_status run_forward(DeviceInfo& dev, const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H, int Sq, int Sk, int D, float scale, int causal, const int32_t* kv_lens, int num_splits,
                        float* o_part, float* lse_part, cudaStream_t s, int kernel = ATTN_KERNEL_AUTO,
                        uint64_t wait_limit_ns = kWaitLimitNs, int selftest_skip_fill = -1) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, B, H, Sq, D)) return ATTN_ERR_CUDA;
  if (Sk > 0) {
    if (!make_map(&mk, k, B, H, Sk, D) || !make_map(&mv, v, B, H, Sk, D)) return ATTN_ERR_CUDA;
  } else {  // never dereferenced: with no keys every unit has zero K tiles
    mk = mq;
    mv = mq;
  }
  const uint64_t n_qtiles = (static_cast<uint64_t>(Sq) + kBQ - 1) / kBQ;
  Params p;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.kv_lens = kv_lens;
  p.B = B;
  p.H = H;
  p.Sq = Sq;
  p.Sk = Sk;
  p.n_qtiles = static_cast<int>(n_qtiles);
  p.head_group = head_group_for(B * H, Sk, D, 2);
  p.num_splits = num_splits;
  p.total_units = static_cast<int>(static_cast<uint64_t>(B) * H * n_qtiles * num_splits);
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.cu_q = nullptr;
  p.cu_k = nullptr;
  p.total_q = 0;
  p.total_k = 0;
  clear_paged(p);
  p.sched = nullptr;
  p.c = static_cast<float>(std::fabs(static_cast<double>(scale)) * 1.4426950408889634);
  p.v_scale = 1.0f;
  p.idesc_qk = idesc_bf16_f32(kBQ, kBK, scale < 0.0f, false);
  p.idesc_pv = idesc_bf16_f32(kBQ, D, false, true);
  p.wait_limit_ns = wait_limit_ns;
  p.selftest_skip_fill = selftest_skip_fill;
#ifndef ATTN_NO_PAIR
  const bool pair =
      kernel == ATTN_KERNEL_TWO_TILE ||
      (kernel == ATTN_KERNEL_AUTO && attn_pair_host::use_pair(B, H, Sq, Sk, D, causal != 0, dev.num_sms, false));
  if (o_part == nullptr && pair) {
    // whole rows: units of two query tiles (attn_fwd_pair_kernel)
    Params pp = p;
    const uint64_t n_pairs = (static_cast<uint64_t>(Sq) + 2 * kBQ - 1) / (2 * kBQ);
    pp.n_qtiles = static_cast<int>(n_pairs);
    pp.total_units = static_cast<int>(static_cast<uint64_t>(B) * H * n_pairs);
    return attn_pair_host::launch(D, causal != 0, false, dev.num_sms, mq, mk, mv, pp, s);
  }
#endif
  if (D == 64) {
    return causal ? launch<64, true>(dev, 0, mq, mk, mv, p, s) : launch<64, false>(dev, 1, mq, mk, mv, p, s);
  }
  return causal ? launch<128, true>(dev, 2, mq, mk, mv, p, s) : launch<128, false>(dev, 3, mq, mk, mv, p, s);
}

#include "attn_bwd.cuh"

}  // namespace

extern "C" {

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Sq, int Sk,
                     int D, float scale, int causal, const int32_t* kv_lens, attn_stream_t stream) {
  attn_status st = check_args(q, k, v, o, lse, B, H, Sq, Sk, D, scale, kv_lens, 1);
  if (st != ATTN_OK || B == 0 || H == 0 || Sq == 0) return st;
  DeviceInfo* dev = nullptr;
  st = device_info(&dev);
  if (st != ATTN_OK) return st;
  return run_forward(*dev, q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, kv_lens, 1, nullptr, nullptr,
                     reinterpret_cast<cudaStream_t>(stream));
}

attn_status attn_fwd_variant(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Sq,
                             int Sk, int D, float scale, int causal, const int32_t* kv_lens, int kernel,
                             attn_stream_t stream) {
  if (kernel < ATTN_KERNEL_AUTO || kernel > ATTN_KERNEL_TWO_TILE) return ATTN_ERR_SHAPE;
  attn_status st = check_args(q, k, v, o, lse, B, H, Sq, Sk, D, scale, kv_lens, 1);
  if (st != ATTN_OK || B == 0 || H == 0 || Sq == 0) return st;
  DeviceInfo* dev = nullptr;
  st = device_info(&dev);
  if (st != ATTN_OK) return st;
  return run_forward(*dev, q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, kv_lens, 1, nullptr, nullptr,
                     reinterpret_cast<cudaStream_t>(stream), kernel);
}

attn_status attn_fwd_fp8_variant(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                 int Sq, int Sk, int D, float scale, int causal, const int32_t* kv_lens,
                                 float q_descale, float k_descale, float v_descale, int v_layout, int kernel,
                                 attn_stream_t stream) {
  if (v_layout != ATTN_V_ROWS && v_layout != ATTN_V_TRANSPOSED) return ATTN_ERR_SHAPE;
  if (kernel < ATTN_KERNEL_AUTO || kernel > ATTN_KERNEL_TWO_TILE) return ATTN_ERR_SHAPE;
  const bool v_rows = v_layout == ATTN_V_ROWS;
  const void* v_t = v;
  if (B < 0 || H < 0 || Sq < 0 || Sk < 0) return ATTN_ERR_SHAPE;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED_D;
  if (!std::isfinite(scale) || !std::isfinite(q_descale) || !std::isfinite(k_descale) || !std::isfinite(v_descale))
    return ATTN_ERR_SCALE;
  const double qk_scale = static_cast<double>(scale) * q_descale * k_descale;
  if (!std::isfinite(static_cast<float>(qk_scale))) return ATTN_ERR_SCALE;
  if (!v_rows && Sk % 16 != 0) return ATTN_ERR_SHAPE;  // V^T rows are Sk bytes: a TMA stride must be a multiple of 16
  if (B == 0 || H == 0 || Sq == 0) return ATTN_OK;
  if (q == nullptr || o == nullptr || lse == nullptr) return ATTN_ERR_NULLPTR;
  if (Sk > 0 && (k == nullptr || v_t == nullptr)) return ATTN_ERR_NULLPTR;
  if (!aligned(q, 16) || !aligned(o, 16) || !aligned(lse, 4)) return ATTN_ERR_ALIGN;
  if (Sk > 0 && (!aligned(k, 16) || !aligned(v_t, 16))) return ATTN_ERR_ALIGN;
  if (kv_lens != nullptr && !aligned(kv_lens, 4)) return ATTN_ERR_ALIGN;
  const uint64_t max_s = static_cast<uint64_t>(Sq > Sk ? Sq : Sk);
  if (static_cast<uint64_t>(H) * max_s * D * 2 >= (1ull << 40)) return ATTN_ERR_SHAPE;
  const uint64_t n_qtiles = (static_cast<uint64_t>(Sq) + kBQ - 1) / kBQ;
  if (static_cast<uint64_t>(B) * H * n_qtiles > 0x7fff0000ull) return ATTN_ERR_SHAPE;
  DeviceInfo* dev = nullptr;
  attn_status st = device_info(&dev);
  if (st != ATTN_OK) return st;
  CUtensorMap mq, mk, mv;
  const uint32_t dbox = static_cast<uint32_t>(D);  // bytes of a row of D
  if (!make_map_e4m3(&mq, q, D, Sq, H, B, dbox, 128)) return ATTN_ERR_CUDA;
  if (Sk > 0) {
    if (!make_map_e4m3(&mk, k, D, Sk, H, B, dbox, 128)) return ATTN_ERR_CUDA;
    if (v_rows ? !make_map_e4m3(&mv, v, D, Sk, H, B, dbox, 128) : !make_map_e4m3(&mv, v_t, Sk, D, H, B, 128, dbox))
      return ATTN_ERR_CUDA;
  } else {  // never dereferenced: with no keys every unit has zero K tiles
    mk = mq;
    mv = mq;
  }
  Params p;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.kv_lens = kv_lens;
  p.B = B;
  p.H = H;
  p.Sq = Sq;
  p.Sk = Sk;
  p.n_qtiles = static_cast<int>(n_qtiles);
  p.head_group = head_group_for(B * H, Sk, D, 1);
  p.num_splits = 1;
  p.total_units = static_cast<int>(static_cast<uint64_t>(B) * H * n_qtiles);
  p.o_part = nullptr;
  p.lse_part = nullptr;
  p.cu_q = nullptr;
  p.cu_k = nullptr;
  p.total_q = 0;
  p.total_k = 0;
  clear_paged(p);
  p.sched = nullptr;
  p.c = static_cast<float>(std::fabs(qk_scale) * 1.4426950408889634);
  p.v_scale = v_descale;
  p.idesc_qk = idesc_e4m3_f32(kBQ, kBK, qk_scale < 0.0);
  p.idesc_pv = idesc_e4m3_f32(kBQ, D, false, v_rows);
  p.v_rows = v_rows ? 1 : 0;
  p.wait_limit_ns = kWaitLimitNs;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (kernel == ATTN_KERNEL_TWO_TILE ||
      (kernel == ATTN_KERNEL_AUTO && attn_pair_host::use_pair(B, H, Sq, Sk, D, causal != 0, dev->num_sms, true))) {
    // units of two query tiles (attn_fwd_pair_kernel), by the E4M3 cost model
    Params pp = p;
    const uint64_t n_pairs = (static_cast<uint64_t>(Sq) + 2 * kBQ - 1) / (2 * kBQ);
    pp.n_qtiles = static_cast<int>(n_pairs);
    pp.total_units = static_cast<int>(static_cast<uint64_t>(B) * H * n_pairs);
    return attn_pair_host::launch(D, causal != 0, true, dev->num_sms, mq, mk, mv, pp, s);
  }
  if (D == 64)
    return causal ? launch<64, true, true>(*dev, 12, mq, mk, mv, p, s) : launch<64, false, true>(*dev, 13, mq, mk, mv, p, s);
  return causal ? launch<128, true, true>(*dev, 4, mq, mk, mv, p, s) : launch<128, false, true>(*dev, 5, mq, mk, mv, p, s);
}

attn_status attn_fwd_fp8_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Sq,
                            int Sk, int D, float scale, int causal, const int32_t* kv_lens, float q_descale,
                            float k_descale, float v_descale, int v_layout, attn_stream_t stream) {
  return attn_fwd_fp8_variant(q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, kv_lens, q_descale, k_descale,
                              v_descale, v_layout, ATTN_KERNEL_AUTO, stream);
}

attn_status attn_fwd_fp8(const void* q, const void* k, const void* v_t, void* o, float* lse, int B, int H, int Sq,
                         int Sk, int D, float scale, int causal, const int32_t* kv_lens, float q_descale,
                         float k_descale, float v_descale, attn_stream_t stream) {
  return attn_fwd_fp8_ex(q, k, v_t, o, lse, B, H, Sq, Sk, D, scale, causal, kv_lens, q_descale, k_descale, v_descale,
                         ATTN_V_TRANSPOSED, stream);
}

attn_status attn_fwd_varlen_variant(const void* q, const void* k, const void* v, void* o, float* lse,
                                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch,
                                    int max_seqlen_q, int total_q, int total_k, int H, int D, float scale, int causal,
                                    uint32_t* tile_counter, int kernel, attn_stream_t stream) {
  if (kernel < ATTN_KERNEL_AUTO || kernel > ATTN_KERNEL_TWO_TILE) return ATTN_ERR_SHAPE;
  if (batch < 0 || max_seqlen_q < 0 || total_q < 0 || total_k < 0 || H < 0) return ATTN_ERR_SHAPE;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED_D;
  if (!std::isfinite(scale)) return ATTN_ERR_SCALE;
  if (batch == 0 || H == 0 || total_q == 0 || max_seqlen_q == 0) return ATTN_OK;
  if (q == nullptr || o == nullptr || lse == nullptr || cu_seqlens_q == nullptr || cu_seqlens_k == nullptr)
    return ATTN_ERR_NULLPTR;
  if (total_k > 0 && (k == nullptr || v == nullptr)) return ATTN_ERR_NULLPTR;
  if (!aligned(q, 16) || !aligned(o, 16) || !aligned(lse, 4) || !aligned(cu_seqlens_q, 4) ||
      !aligned(cu_seqlens_k, 4))
    return ATTN_ERR_ALIGN;
  if (total_k > 0 && (!aligned(k, 16) || !aligned(v, 16))) return ATTN_ERR_ALIGN;
  if (tile_counter != nullptr && !aligned(tile_counter, 8)) return ATTN_ERR_ALIGN;
  const uint64_t max_t = static_cast<uint64_t>(total_q > total_k ? total_q : total_k);
  if (max_t * H * D * 2 >= (1ull << 40)) return ATTN_ERR_SHAPE;
  const uint64_t n_qtiles = (static_cast<uint64_t>(max_seqlen_q) + kBQ - 1) / kBQ;
  if (static_cast<uint64_t>(batch) * H * n_qtiles > 0x7fff0000ull) return ATTN_ERR_SHAPE;
  DeviceInfo* dev = nullptr;
  attn_status st = device_info(&dev);
  if (st != ATTN_OK) return st;
  CUtensorMap mq, mk, mv;
  if (!make_map_packed(&mq, q, H, total_q, D)) return ATTN_ERR_CUDA;
  if (total_k > 0) {
    if (!make_map_packed(&mk, k, H, total_k, D) || !make_map_packed(&mv, v, H, total_k, D)) return ATTN_ERR_CUDA;
  } else {  // never dereferenced: with no keys every unit has zero K tiles
    mk = mq;
    mv = mq;
  }
  Params p = packed_params(o, lse, cu_seqlens_q, batch, max_seqlen_q, total_q, H, D, scale);
  p.cu_k = cu_seqlens_k;
  p.total_k = total_k;
  // claimed units balance ragged non-causal batches (measured +18 %); causal
  // batches keep the longest-first snake deal, since claiming them in
  // longest-first order walks through the empty high query tiles of the short
  // sequences one atomic at a time (measured 8 % slower)
  p.sched = causal ? nullptr : tile_counter;
  // Units of two query tiles of one (sequence, head) (attn_fwd_pair_kernel)
  // whenever a sequence may hold more than one query tile, claimed from the
  // counter when it is given (causal too), in longest-first order over all
  // heads (measured on the packed workload, 32 sequences U[1,4096]: causal
  // 1063 TFLOP/s claimed and 967 dealt, against 942 on the one-tile kernel;
  // by head groups, as the one-tile kernel orders them, 984; non-causal
  // claimed 1350-1409 against 1238).
  if (kernel == ATTN_KERNEL_TWO_TILE || (kernel == ATTN_KERNEL_AUTO && max_seqlen_q > kBQ)) {
    Params pp = p;
    pp.sched = tile_counter;
    pp.head_group = batch * H;
    const uint64_t n_pairs = (static_cast<uint64_t>(max_seqlen_q) + 2 * kBQ - 1) / (2 * kBQ);
    pp.n_qtiles = static_cast<int>(n_pairs);
    pp.total_units = static_cast<int>(static_cast<uint64_t>(batch) * H * n_pairs);
    return attn_pair_host::launch(D, causal != 0, false, dev->num_sms, mq, mk, mv, pp,
                                  reinterpret_cast<cudaStream_t>(stream));
  }
  return launch_any(*dev, D, causal != 0, mq, mk, mv, p, reinterpret_cast<cudaStream_t>(stream));
}

attn_status attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch, int max_seqlen_q,
                            int total_q, int total_k, int H, int D, float scale, int causal, uint32_t* tile_counter,
                            attn_stream_t stream) {
  return attn_fwd_varlen_variant(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, batch, max_seqlen_q, total_q, total_k, H,
                                 D, scale, causal, tile_counter, ATTN_KERNEL_AUTO, stream);
}

attn_status attn_fwd_paged_variant(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                                   const int32_t* cu_seqlens_q, const int32_t* seqlens_k,
                                   const int32_t* block_table, int batch, int max_seqlen_q, int total_q,
                                   int num_pages, int page_size, int max_pages_per_seq, int H, int D, float scale,
                                   int causal, uint32_t* tile_counter, int kernel, attn_stream_t stream) {
  if (kernel < ATTN_KERNEL_AUTO || kernel > ATTN_KERNEL_TWO_TILE) return ATTN_ERR_SHAPE;
  if (batch < 0 || max_seqlen_q < 0 || total_q < 0 || H < 0) return ATTN_ERR_SHAPE;
  if (num_pages < 1 || max_pages_per_seq < 1 || page_size < 64 || page_size % 64 != 0) return ATTN_ERR_SHAPE;
  if (static_cast<uint64_t>(num_pages) * page_size + 64 > 0x7fffffffull ||
      static_cast<uint64_t>(max_pages_per_seq) * page_size > 0x7fffffffull)
    return ATTN_ERR_SHAPE;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED_D;
  if (!std::isfinite(scale)) return ATTN_ERR_SCALE;
  if (batch == 0 || H == 0 || total_q == 0 || max_seqlen_q == 0) return ATTN_OK;
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || o == nullptr || lse == nullptr ||
      cu_seqlens_q == nullptr || seqlens_k == nullptr || block_table == nullptr)
    return ATTN_ERR_NULLPTR;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(cu_seqlens_q, 4) || !aligned(seqlens_k, 4) || !aligned(block_table, 4) ||
      (tile_counter != nullptr && !aligned(tile_counter, 8)))
    return ATTN_ERR_ALIGN;
  const uint64_t cache_tokens = static_cast<uint64_t>(num_pages) * page_size;
  const uint64_t max_t = cache_tokens > static_cast<uint64_t>(total_q) ? cache_tokens : total_q;
  if (max_t * H * D * 2 >= (1ull << 40)) return ATTN_ERR_SHAPE;
  const uint64_t n_qtiles = (static_cast<uint64_t>(max_seqlen_q) + kBQ - 1) / kBQ;
  if (static_cast<uint64_t>(batch) * H * n_qtiles > 0x7fff0000ull) return ATTN_ERR_SHAPE;
  DeviceInfo* dev = nullptr;
  attn_status st = device_info(&dev);
  if (st != ATTN_OK) return st;
  CUtensorMap mq, mk, mv;
  if (!make_map_packed(&mq, q, H, total_q, D) ||
      !make_map_packed(&mk, k_cache, H, static_cast<int>(cache_tokens), D, 64) ||
      !make_map_packed(&mv, v_cache, H, static_cast<int>(cache_tokens), D, 64))
    return ATTN_ERR_CUDA;
  Params p = packed_params(o, lse, cu_seqlens_q, batch, max_seqlen_q, total_q, H, D, scale);
  p.block_table = block_table;
  p.seqlens_k = seqlens_k;
  p.page_size = page_size;
  p.max_pages = max_pages_per_seq;
  p.num_pages = num_pages;
  p.cache_tokens = static_cast<int>(cache_tokens);
  p.sched = causal ? nullptr : tile_counter;  // as attn_fwd_varlen
  // causal paged batches keep the longest-first order over all heads: the
  // head groups that help the packed batch (+9 %) cost this one 5 % (measured)
  p.head_group = batch * H;
  if (kernel == ATTN_KERNEL_TWO_TILE || (kernel == ATTN_KERNEL_AUTO && max_seqlen_q > kBQ)) {
    // units of two query tiles of one (sequence, head) (attn_fwd_pair_kernel),
    // claimed from the counter when it is given (measured on the paged
    // workload, causal: 1045 TFLOP/s claimed and 965 dealt, against 807-813
    // on the one-tile kernel)
    Params pp = p;
    pp.sched = tile_counter;
    const uint64_t n_pairs = (static_cast<uint64_t>(max_seqlen_q) + 2 * kBQ - 1) / (2 * kBQ);
    pp.n_qtiles = static_cast<int>(n_pairs);
    pp.total_units = static_cast<int>(static_cast<uint64_t>(batch) * H * n_pairs);
    return attn_pair_host::launch(D, causal != 0, false, dev->num_sms, mq, mk, mv, pp,
                                  reinterpret_cast<cudaStream_t>(stream));
  }
  return launch_any(*dev, D, causal != 0, mq, mk, mv, p, reinterpret_cast<cudaStream_t>(stream));
}

attn_status attn_fwd_paged(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                           const int32_t* cu_seqlens_q, const int32_t* seqlens_k, const int32_t* block_table,
                           int batch, int max_seqlen_q, int total_q, int num_pages, int page_size,
                           int max_pages_per_seq, int H, int D, float scale, int causal, uint32_t* tile_counter,
                           attn_stream_t stream) {
  return attn_fwd_paged_variant(q, k_cache, v_cache, o, lse, cu_seqlens_q, seqlens_k, block_table, batch,
                                max_seqlen_q, total_q, num_pages, page_size, max_pages_per_seq, H, D, scale, causal,
                                tile_counter, ATTN_KERNEL_AUTO, stream);
}

size_t attn_fwd_splitkv_workspace_size(int B, int H, int Sq, int D, int num_splits) {
  if (B < 0 || H < 0 || Sq < 0 || (D != 64 && D != 128) || num_splits < 1 || num_splits > kMaxSplits) return 0;
  return splitkv_bytes(B, H, Sq, D, num_splits, nullptr);
}

// Equal ranges matter because the slowest range sets the time: on 8 query
// blocks against 32768 keys (256 tiles) on 152 SMs, 16 equal ranges took
// 45.3 us and 19 ranges of 13-14 tiles 46.4 us (merge included).
int attn_fwd_splitkv_suggest_splits(int B, int H, int Sq, int Sk, int num_sms) {
  if (B < 0 || H < 0 || Sq < 0 || Sk < 0 || num_sms < 1) return 0;
  const int64_t units = static_cast<int64_t>(B) * H * ((static_cast<int64_t>(Sq) + kBQ - 1) / kBQ);
  if (units == 0 || units >= num_sms) return 1;
  const int64_t tiles = Sk > 0 ? (static_cast<int64_t>(Sk) + kBK - 1) / kBK : 1;
  int64_t s_max = num_sms / units;
  if (s_max > tiles) s_max = tiles;
  if (s_max > kMaxSplits) s_max = kMaxSplits;
  if (s_max < 1) s_max = 1;
  int64_t even = 1;
  for (int64_t s = s_max; s >= 1; --s)
    if (tiles % s == 0) {
      even = s;
      break;
    }
  return static_cast<int>(2 * even >= s_max ? even : s_max);
}

attn_status attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Sq,
                             int Sk, int D, float scale, int causal, const int32_t* kv_lens, int num_splits,
                             void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  attn_status st = check_args(q, k, v, o, lse, B, H, Sq, Sk, D, scale, kv_lens, num_splits);
  if (st != ATTN_OK || B == 0 || H == 0 || Sq == 0) return st;
  size_t lse_off = 0;
  const size_t need = splitkv_bytes(B, H, Sq, D, num_splits, &lse_off);
  if (workspace == nullptr) return ATTN_ERR_NULLPTR;
  if (!aligned(workspace, 256)) return ATTN_ERR_ALIGN;
  if (workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  st = device_info(&dev);
  if (st != ATTN_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* o_part = static_cast<float*>(workspace);
  float* lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + lse_off);
  st = run_forward(*dev, q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, kv_lens, num_splits, o_part, lse_part, s);
  if (st != ATTN_OK) return st;
  return launch_merge(*dev, o_part, lse_part, num_splits, static_cast<long long>(B) * H * Sq, D, o, lse, s);
}

attn_status attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                     int Sq, int Sk, int D, float scale, int causal, const int32_t* kv_lens,
                                     int num_splits, attn_stream_t stream) {
  attn_status st = check_args(q, k, v, o, lse, B, H, Sq, Sk, D, scale, kv_lens, num_splits);
  if (st != ATTN_OK || B == 0 || H == 0 || Sq == 0) return st;
  if (splitkv_bytes(B, H, Sq, D, num_splits, nullptr) > static_cast<size_t>(ATTN_SPLITKV_SCRATCH_BYTES))
    return ATTN_ERR_WORKSPACE;
  DeviceInfo* dev = nullptr;
  st = device_info(&dev);
  if (st != ATTN_OK) return st;
  // The array exists once per CUDA context, and in host code its name is
  // only a stand-in: the device address is looked up in the current context
  // on every call (a host-side query that allocates nothing), so a context
  // made current after a reset or by the caller is never given another
  // context's address.
  void* scratch = nullptr;
  if (cudaGetSymbolAddress(&scratch, g_splitkv_scratch) != cudaSuccess || scratch == nullptr) return ATTN_ERR_CUDA;
  return attn_fwd_splitkv(q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, kv_lens, num_splits, scratch,
                          static_cast<size_t>(ATTN_SPLITKV_SCRATCH_BYTES), stream);
}

attn_status attn_lse_merge(const float* o_parts, const float* lse_parts, int num_parts, void* o, float* lse,
                           long long rows, int D, attn_stream_t stream) {
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED_D;
  if (num_parts < 1 || rows < 0) return ATTN_ERR_SHAPE;
  if (rows == 0) return ATTN_OK;
  if (o_parts == nullptr || lse_parts == nullptr || o == nullptr || lse == nullptr) return ATTN_ERR_NULLPTR;
  if (!aligned(o_parts, 16) || !aligned(lse_parts, 4) || !aligned(o, 8) || !aligned(lse, 4)) return ATTN_ERR_ALIGN;
  DeviceInfo* dev = nullptr;
  attn_status st = device_info(&dev);
  if (st != ATTN_OK) return st;
  return launch_merge(*dev, o_parts, lse_parts, num_parts, rows, D, o, lse, reinterpret_cast<cudaStream_t>(stream));
}

size_t attn_bwd_workspace_size(int B, int H, int Sq) {
  if (B < 0 || H < 0 || Sq < 0) return 0;
  return bwd_delta_bytes(B, H, Sq);
}

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                     void* dq, void* dk, void* dv, int B, int H, int Sq, int Sk, int D, float scale, int causal,
                     const int32_t* kv_lens, void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  attn_status st = check_args(q, k, v, o, lse, B, H, Sq, Sk, D, scale, kv_lens, 1);
  if (st != ATTN_OK) return st;
  if (B == 0 || H == 0 || (Sq == 0 && Sk == 0)) return ATTN_OK;
  if (Sq > 0 && (dout == nullptr || dq == nullptr)) return ATTN_ERR_NULLPTR;
  if (Sk > 0 && (dk == nullptr || dv == nullptr)) return ATTN_ERR_NULLPTR;
  if (Sq > 0 && (!aligned(dout, 16) || !aligned(dq, 16))) return ATTN_ERR_ALIGN;
  if (Sk > 0 && (!aligned(dk, 16) || !aligned(dv, 16))) return ATTN_ERR_ALIGN;
  if (Sq > 0 && Sk > 0) {
    if (workspace == nullptr) return ATTN_ERR_NULLPTR;
    if (!aligned(workspace, 256)) return ATTN_ERR_ALIGN;
    if (workspace_bytes < bwd_delta_bytes(B, H, Sq)) return ATTN_ERR_WORKSPACE;
  }
  DeviceInfo* dev = nullptr;
  st = device_info(&dev);
  if (st != ATTN_OK) return st;
  return run_backward(*dev, q, k, v, o, dout, lse, dq, dk, dv, B, H, Sq, Sk, D, scale, causal, kv_lens,
                      static_cast<float*>(workspace), reinterpret_cast<cudaStream_t>(stream));
}

const char* attn_get_error_string(attn_status status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_NULLPTR: return "a required pointer is NULL";
    case ATTN_ERR_ALIGN: return "q/k/v/o must be 16-byte aligned, lse and kv_lens 4-byte aligned";
    case ATTN_ERR_SHAPE: return "invalid or too large B/H/Sq/Sk/num_splits";
    case ATTN_ERR_UNSUPPORTED_D: return "head dimension D must be 64 or 128";
    case ATTN_ERR_SCALE: return "scale must be finite";
    case ATTN_ERR_CUDA: return "a CUDA call failed";
    case ATTN_ERR_DEVICE_TIMEOUT: return "a device-side wait gave up (kernel aborted its work)";
    case ATTN_ERR_UNSUPPORTED_DEVICE: return "the current device is not an sm_103 (GB300) GPU";
    case ATTN_ERR_WORKSPACE: return "workspace smaller than attn_fwd_splitkv_workspace_size()";
  }
  return "unknown status";
}

attn_status attn_check_device_status(attn_stream_t stream, uint32_t* site) {
  if (site != nullptr) *site = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
  // each translation unit's kernels report into their own status word
  uint32_t host[3] = {0, 0, 0};
  if (cudaMemcpyFromSymbol(host, g_attn_status, sizeof(host)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (host[0] != 0) {
    const uint32_t zero[3] = {0, 0, 0};
    if (cudaMemcpyToSymbol(g_attn_status, zero, sizeof(zero)) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  uint32_t pair[3] = {0, 0, 0};
  if (attn_pair_host::status_read_clear(pair) != ATTN_OK) return ATTN_ERR_CUDA;
  if (host[0] == 0 && pair[0] == 0) return ATTN_OK;
  if (site != nullptr) *site = host[0] != 0 ? host[1] : pair[1];
  return ATTN_ERR_DEVICE_TIMEOUT;
}

attn_status attn_selftest_wait_timeout(int64_t limit_ns, attn_stream_t stream) {
  if (limit_ns < 1 || limit_ns > 2000000000LL) return ATTN_ERR_SHAPE;
  DeviceInfo* dev = nullptr;
  attn_status st = device_info(&dev);
  if (st != ATTN_OK) return st;
  wait_timeout_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint64_t>(limit_ns));
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_selftest_fwd_abort(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                    int Sq, int Sk, int D, float scale, int causal, const int32_t* kv_lens,
                                    int kernel, int skip_fill, int64_t limit_ns, attn_stream_t stream) {
  if (kernel < ATTN_KERNEL_AUTO || kernel > ATTN_KERNEL_TWO_TILE) return ATTN_ERR_SHAPE;
  attn_status st = check_args(q, k, v, o, lse, B, H, Sq, Sk, D, scale, kv_lens, 1);
  if (st != ATTN_OK) return st;
  if (limit_ns < 1000 || limit_ns > 2000000000LL || skip_fill < 0) return ATTN_ERR_SHAPE;
  // block 0 must have a K fill with that index: its first unit's tiles
  if (B == 0 || H == 0 || Sq == 0 || Sk == 0) return ATTN_ERR_SHAPE;
  DeviceInfo* dev = nullptr;
  st = device_info(&dev);
  if (st != ATTN_OK) return st;
  return run_forward(*dev, q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, kv_lens, 1, nullptr, nullptr,
                     reinterpret_cast<cudaStream_t>(stream), kernel, static_cast<uint64_t>(limit_ns), skip_fill);
}

attn_status attn_selftest_launch_floor(int grid, int D, int mode, attn_stream_t stream) {
  if (grid < 1 || grid > 65535 || mode < 0 || mode > 1) return ATTN_ERR_SHAPE;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED_D;
  DeviceInfo* dev = nullptr;
  attn_status st = device_info(&dev);
  if (st != ATTN_OK) return st;
  const int smem = D == 64 ? Geo<64>::kSmemBytes : Geo<128>::kSmemBytes;
  // both sizes exceed half of an SM's shared memory: one block per SM
  static_assert(2 * Geo<128>::kSmemBytes > 233472 && 2 * Geo<64>::kSmemBytes > 233472, "one block per SM");
  const int idx = D == 64 ? 10 : 11;
  if (!dev->smem_set[idx].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(launch_floor_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Geo<64>::kSmemBytes > Geo<128>::kSmemBytes ? Geo<64>::kSmemBytes : Geo<128>::kSmemBytes) !=
        cudaSuccess)
      return ATTN_ERR_CUDA;
    dev->smem_set[idx].store(true, std::memory_order_release);
  }
  launch_floor_kernel<<<grid, kThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(mode);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int64_t attn_fwd_pair_schedule(int B, int H, int Sq, int Sk, int head_group, int grid, uint8_t* owner,
                               int64_t max_units) {
  return attn_pair_host::build_schedule(B, H, Sq, Sk, head_group, grid, owner, max_units);
}

int attn_fwd_kernel_choice(int B, int H, int Sq, int Sk, int D, int causal, int num_sms) {
  if (B < 0 || H < 0 || Sq < 0 || Sk < 0 || num_sms < 0 || (D != 64 && D != 128)) return -1;
  return attn_pair_host::use_pair(B, H, Sq, Sk, D, causal != 0, num_sms, false) ? 1 : 0;
}

int attn_fwd_fp8_kernel_choice(int B, int H, int Sq, int Sk, int D, int causal, int num_sms) {
  if (B < 0 || H < 0 || Sq < 0 || Sk < 0 || num_sms < 0 || (D != 64 && D != 128)) return -1;
  return attn_pair_host::use_pair(B, H, Sq, Sk, D, causal != 0, num_sms, true) ? 1 : 0;
}

int attn_abi_version(void) { return ATTN_ABI_VERSION; }

}  // extern "C"
