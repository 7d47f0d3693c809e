// The forward with two query tiles per work unit.
//
// Same operation as attn_fwd_kernel (softmax(scale * Q K^T + mask) V and the
// row LSE; "Kernel Fusion and the Memory Wall", section "FlashAttention: avoid
// the full score matrix", and the tile loop of "Attention softmax fusion"), for
// padded [B, H, S, D] batches without key ranges (bf16 or E4M3, the FP8
// template parameter) and for packed and paged bf16 batches (the PACKED
// template parameter, instantiations of their own).  A translation unit of its
// own (with the shared parameters, waits and unit order of attn_common.cuh),
// so that its code leaves the register allocation of attn_fwd.cu's kernels
// untouched: compiled into one file with them, it cost two of those kernels a
// register spill.
//
// A work unit is 256 query rows of one (b, h) (packed: of one sequence and
// head): tiles A (rows q0 .. q0 + 127) and B (q0 + 128 .. q0 + 255), which
// share every K/V tile the producer loads.
// Each tile has one softmax warpgroup with ONE thread per row (warps 0-3: A,
// warps 4-7: B), so a row's max and sum never leave its thread: no barrier,
// no exchange.  The two tiles' work interleaves on the tensor pipe: while
// the softmax of A works on S_A, the pipe computes S_B = Q_B K^T and the
// previous P_B V, and the other way round.
//
//   warps 0-3  softmax of tile A (thread = row)
//   warps 4-7  softmax of tile B
//   warp 8     TMA producer of the unit queue, the Q pair and the K/V ring (one lane)
//   warp 9     TMEM owner; issues S_x = Q_x K^T for x = A, B
//   warp 10    issues O_x += P_x V for x = A, B
//   warp 11    idle
//
// Tensor Memory (512 columns): S_A [0,128), S_B [128,256), O_A [256, 256+D),
// O_B [256+D, 256+2D).  P_x (bf16 pairs in 64 columns; E4M3, four a word, in
// 32) is written over the first columns of S_x once the softmax has read S_x;
// S_x is written again only after the P V of its previous tile has consumed
// P_x (the QK^T issuer waits for that product's commit).  So when the
// softmax of x sees a new S_x, the P V of the previous tile has completed and
// O_x is stable: a rescale of O_x never waits.
//
// Every wait is bounded, as in attn_fwd_kernel; a wait that gives up records
// its site and raises the block's abort flag, and every role drains what it
// has in flight, frees TMEM and returns.  The softmax threads never use a
// named barrier, so no role can be left waiting for another that has left.

#include <algorithm>
#include <atomic>
#include <cstring>
#include <functional>
#include <mutex>
#include <queue>
#include <utility>
#include <vector>

#include "attn_common.cuh"
#include "attn_pair_host.h"

using namespace attn_sm103;

namespace {

template <int D, bool FP8>
struct GeoPair {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kElem = FP8 ? 1 : 2;           // bytes per element of Q, K, V
  static constexpr int kRowBytes = D * kElem;         // one row of a Q or K tile (and of V in rows)
  static constexpr int kTileBytes = 128 * kRowBytes;  // one Q, K or V tile (128 rows)
  // Rows of 128 bytes (bf16 D = 64, E4M3 D = 128) or 256 bytes (bf16 D =
  // 128, two 64-column chunks) use the 128-byte swizzle; the 64-byte rows of
  // E4M3 at D = 64 the 64-byte swizzle (8-row atoms of 64 bytes, 512 apart).
  static constexpr bool kSw64 = kRowBytes == 64;
  static constexpr int kChunkBytes = kSw64 ? 128 * 64 : 128 * 128;  // 128 rows of one swizzle column
  static constexpr int kChunks = kSw64 ? 1 : kRowBytes / 128;
  static constexpr int kChunkElems = kSw64 ? 64 : 128 / kElem;      // elements per row of a chunk
  static constexpr uint32_t kSwMode = kSw64 ? kSmemSwizzle64B : kSmemSwizzle128B;
  static constexpr uint32_t kSbo = kSw64 ? 512 : 1024;               // 8-row groups of a chunk
  static constexpr int kKSteps = kRowBytes / 32;      // QK^T instructions: 32 bytes of D each
  static constexpr int kPCols = 128 * kElem / 4;      // TMEM columns of one tile's P (128 keys)
  static constexpr int kOffQ = 1024;                  // after the control block
  static constexpr int kOffRing = kOffQ + 2 * kTileBytes;
  // E4M3 at D = 64 keeps an unused tile-sized pad after the ring, as the
  // one-tile kernel does, so that no read of the last slot leaves the block
  static constexpr int kPadBytes = kSw64 ? kTileBytes : 0;
  // as many K/V slots as the 227 KB a block may use leave, at most 16 (bf16
  // D = 128: 5, bf16 D = 64 and E4M3 D = 128: 12, E4M3 D = 64: 16)
  static constexpr int kSlotsFit = (232448 - kOffRing - kPadBytes) / kTileBytes;
  static constexpr int kSlots = kSlotsFit < 16 ? kSlotsFit : 16;
  static constexpr int kSmemBytes = kOffRing + kSlots * kTileBytes + kPadBytes;
  static_assert(kSlots >= 2 && kSlots <= 16, "ring depth");
  static_assert(2 * kSmemBytes > 233472, "one block per SM (the TMEM allocation is the whole of it)");
  static constexpr uint32_t kTmemS = 0;               // + 128 * x
  static constexpr uint32_t kTmemO = 256;             // + D * x
  // One ring of alternating K and V tiles, as attn_fwd_kernel's padded layout
  // (position p = 2 t (+1 for V) in slot p % kSlots; one full barrier per
  // slot and kind; an odd depth alternates kinds within a slot).
  struct Fill {
    uint32_t slot, full_use, empty_use;
  };
  static __device__ __forceinline__ Fill fill_of(uint32_t t, bool is_v) {
    const uint32_t pos = 2 * t + (is_v ? 1u : 0u);
    return {pos % kSlots, (kSlots & 1) ? (pos / kSlots) >> 1 : pos / kSlots, pos / kSlots};
  }
};

struct CtrlPair {
  uint64_t q_full, q_empty;
  uint64_t k_full[16], v_full[16], kv_empty[16];
  uint64_t s_full[2], p_full[2], p_free[2], o_full[2];  // per query tile
  uint64_t qk_issued_a;  // one phase per S_A = Q_A K^T issued (orders the tensor pipe's queue)
  uint64_t uq_full[kUnitQ], uq_empty[kUnitQ];
  int unit_q[kUnitQ];
  uint64_t drain[2];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(CtrlPair) <= 1024, "control block");

struct UnitPair {
  int b, h;
  int q0;       // first row of tile A within its sequence
  int rows[2];  // rows of tiles A and B that exist (0 .. 128)
  int kv;       // valid keys of the batch entry
  int n[2];     // K tiles tile A / B processes
  int n_max;
  int q_tok0;   // packed mode: token of tile A's first row
  int k_tok0;   // packed mode: token of the sequence's first key
};

// A static deal of the causal units to the blocks, computed on the host
// (attn_pair_host::build_schedule: longest processing time first, from a
// cost model of each unit) and passed by value with the launch: byte t of
// `owner` is the block that runs unit t of the units' order; n == 0: the
// round-robin deal of unit_at instead.  The non-causal kernel's units are all
// of one length and take the round-robin deal (a one-word placeholder).
constexpr int kSchedMaxUnits = 4096;
template <bool ON>
struct UnitSched {
  int n;
  uint32_t owner[ON ? kSchedMaxUnits / 4 : 1];
};

// Rows, keys and tile counts of a packed unit (u.b, u.h, u.q0 set): the
// sequence's query and key ranges come from the offsets (clamped so that any
// content stays in bounds), paged keys from the sequence's key count.  Kept
// apart from the padded decode, whose code it would otherwise perturb
// (measured: 2.4 % on the padded forward).
template <bool CAUSAL>
__device__ __forceinline__ void packed_extent(const Params& p, UnitPair& u) {
  const int qs = min(max(__ldg(p.cu_q + u.b), 0), p.total_q);
  const int qe = min(max(__ldg(p.cu_q + u.b + 1), qs), p.total_q);
  const int q_len = qe - qs;
  u.q_tok0 = qs + u.q0;
  int kv;
  if (p.block_table != nullptr) {  // paged keys: looked up page by page
    kv = min(max(__ldg(p.seqlens_k + u.b), 0), p.max_pages * p.page_size);
    u.k_tok0 = 0;
  } else {
    const int ks = min(max(__ldg(p.cu_k + u.b), 0), p.total_k);
    const int ke = min(max(__ldg(p.cu_k + u.b + 1), ks), p.total_k);
    kv = ke - ks;
    u.k_tok0 = ks;
  }
  u.kv = kv;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    const int q0x = u.q0 + kBQ * x;
    u.rows[x] = max(min(kBQ, q_len - q0x), 0);
    int lim = kv;
    if (CAUSAL) lim = min(lim, q0x + u.rows[x]);
    u.n[x] = u.rows[x] > 0 ? (lim + kBK - 1) / kBK : 0;
  }
  u.n_max = max(u.n[0], u.n[1]);
}

// Unit t: (b, h, pair of query tiles), ordered as attn_fwd_kernel's units
// (Params::n_qtiles counts tile pairs per head here).
template <bool CAUSAL, bool PACKED>
__device__ __forceinline__ UnitPair decode_pair(const Params& p, int t) {
  UnitPair u;
  int pr, bh;
  if (CAUSAL) {  // head groups, longest units first within a group (see decode_unit)
    const int grp = p.fd_group_units.div(t);
    const int w = t - grp * p.head_group * p.n_qtiles;
    const FastDiv& fh = grp == p.last_group ? p.fd_last_heads : p.fd_group_heads;
    const int wq = fh.div(w);
    pr = p.n_qtiles - 1 - wq;
    bh = grp * p.head_group + (w - wq * static_cast<int>(fh.d));
  } else {
    bh = p.fd_qtiles.div(t);
    pr = t - bh * p.n_qtiles;
  }
  u.b = p.fd_H.div(bh);
  u.h = bh - u.b * p.H;
  u.q0 = pr * (2 * kBQ);
  if constexpr (PACKED) {
    packed_extent<CAUSAL>(p, u);
    return u;
  }
  int kv = p.Sk;
  if (p.kv_lens != nullptr) kv = min(max(__ldg(p.kv_lens + u.b), 0), p.Sk);
  u.kv = kv;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    const int q0x = u.q0 + kBQ * x;
    u.rows[x] = max(min(kBQ, p.Sq - q0x), 0);
    int lim = kv;
    if (CAUSAL) lim = min(lim, q0x + u.rows[x]);  // last row of the tile + 1
    u.n[x] = u.rows[x] > 0 ? (lim + kBK - 1) / kBK : 0;
  }
  u.n_max = max(u.n[0], u.n[1]);
  return u;
}

// p = 2^(s*c - mb) for a thread's 128 scores, packed IN PLACE: bf16 pairs
// (pair e to sp[e]) or, FP8, four E4M3 values a word (pairs 2 w and 2 w + 1
// to sp[w]); each word goes to an index whose scores were already read.
// Masked columns (>= climit) give 0.  Returns the fp32 sum of the unrounded
// terms, and in part_max the quantity the caller's growth test bounds: for
// FP8 the largest of the four 32-column partial sums (a term above the bound
// puts its part's sum above it; over a whole row of 128 terms the sum of
// ordinary terms crossed the E4M3 bound, 2^8.5, on most tiles), for bf16
// (bound 2^16) the sum itself.
template <bool MASKED, bool FP8>
__device__ __forceinline__ float row_exp128(uint32_t (&sp)[128], float c, float mb, int climit, float& part_max) {
  const uint64_t c2 = f2_pack(c, c);
  const uint64_t nmb2 = f2_pack(-mb, -mb);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};  // FP8: one per 32 columns; bf16: interleaved
  float pprev0 = 0.0f, pprev1 = 0.0f;  // FP8: the previous pair, packed with the next
#pragma unroll
  for (int e = 0; e < 64; ++e) {
    const int col = 2 * e;
    float x0, x1;
    f2_unpack(f2_fma(f2_pack(u2f(sp[col]), u2f(sp[col + 1])), c2, nmb2), x0, x1);
    float p0 = ex2_approx(x0);
    float p1 = ex2_approx(x1);
    if (MASKED) {
      p0 = (col < climit) ? p0 : 0.0f;
      p1 = (col + 1 < climit) ? p1 : 0.0f;
    }
    const int a = FP8 ? (e >> 4) : (e & 3);
    acc[a] = f2_add(acc[a], f2_pack(p0, p1));
    if constexpr (FP8) {
      if (e & 1) sp[e >> 1] = pack_e4m3x4(pprev0, pprev1, p0, p1);
      pprev0 = p0;
      pprev1 = p1;
    } else {
      sp[e] = pack_bf16x2(p0, p1);
    }
  }
  if constexpr (FP8) {
    float part[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float lo, hi;
      f2_unpack(acc[q], lo, hi);
      part[q] = lo + hi;
    }
    // (a NaN part must reach part_max, so that the caller's test fails as
    // it would on the sum: fmaxf would drop it)
    part_max = part[0];
#pragma unroll
    for (int q = 1; q < 4; ++q) part_max = (part[q] > part_max || part[q] != part[q]) ? part[q] : part_max;
    return (part[0] + part[1]) + (part[2] + part[3]);
  } else {
    const uint64_t a01 = f2_add(acc[0], acc[1]);
    const uint64_t a23 = f2_add(acc[2], acc[3]);
    float lo, hi;
    f2_unpack(f2_add(a01, a23), lo, hi);
    part_max = lo + hi;
    return part_max;
  }
}

// Maximum of a thread's 128 raw scores (columns >= climit excluded when MASKED).
template <bool MASKED>
__device__ __forceinline__ float row_max128(const uint32_t (&sp)[128], int climit) {
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int col = 0; col < 128; col += 2) {
    float x0 = u2f(sp[col]);
    float x1 = u2f(sp[col + 1]);
    if (MASKED) {
      x0 = (col < climit) ? x0 : -INFINITY;
      x1 = (col + 1 < climit) ? x1 : -INFINITY;
    }
    m4[(col >> 1) & 3] = max3(m4[(col >> 1) & 3], x0, x1);
  }
  return fmaxf(max3(m4[0], m4[1], m4[2]), m4[3]);
}

// A thread's 128 scores of S at TMEM address tS (4 loads of 32 columns).
__device__ __forceinline__ void load_s128(uint32_t tS, uint32_t (&sp)[128]) {
  uint32_t(&a)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sp[0]);
  uint32_t(&b)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sp[32]);
  uint32_t(&c)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sp[64]);
  uint32_t(&d)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sp[96]);
  tmem_ld_32x32b_x32(tS, a);
  tmem_ld_32x32b_x32(tS + 32, b);
  tmem_ld_32x32b_x32(tS + 64, c);
  tmem_ld_32x32b_x32(tS + 96, d);
  tmem_ld_wait_x32(a);
  tmem_ld_wait_x32(b);
  tmem_ld_wait_x32(c);
  tmem_ld_wait_x32(d);
}

template <int D, bool CAUSAL, bool FP8, bool PACKED>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_pair_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                         const __grid_constant__ CUtensorMap map_v, const Params p,
                         const __grid_constant__ UnitSched<CAUSAL> sched) {
  using G = GeoPair<D, FP8>;
  using PR = Prec<FP8>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = smem_addr(smem_raw);
  CtrlPair& ctl = *reinterpret_cast<CtrlPair*>(smem_raw);
  volatile int* abort_flag = &ctl.abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // the swizzle atoms need 1024-byte aligned tiles and the layout has no slack
  if ((base & 1023u) != 0u) {
    if (threadIdx.x == 0) record_give_up(kSiteAlign);
    return;
  }
  const uint32_t bar_q_full = smem_addr(&ctl.q_full);
  const uint32_t bar_q_empty = smem_addr(&ctl.q_empty);
  const uint32_t bar_k_full0 = smem_addr(&ctl.k_full[0]);
  const uint32_t bar_v_full0 = smem_addr(&ctl.v_full[0]);
  const uint32_t bar_kv_empty0 = smem_addr(&ctl.kv_empty[0]);
  const uint32_t bar_s_full0 = smem_addr(&ctl.s_full[0]);   // + 8 * x
  const uint32_t bar_p_full0 = smem_addr(&ctl.p_full[0]);
  const uint32_t bar_p_free0 = smem_addr(&ctl.p_free[0]);
  const uint32_t bar_o_full0 = smem_addr(&ctl.o_full[0]);
  const uint32_t bar_uq_full0 = smem_addr(&ctl.uq_full[0]);
  const uint32_t bar_uq_empty0 = smem_addr(&ctl.uq_empty[0]);
  volatile int* unit_q = ctl.unit_q;

  if (warp == 0) {
    if (lane < G::kSlots) {
      mbar_init(bar_k_full0 + 8 * lane, 1);
      mbar_init(bar_v_full0 + 8 * lane, 1);
      mbar_init(bar_kv_empty0 + 8 * lane, 1);
    } else if (lane >= 16 && lane < 18) {
      const int x = lane - 16;
      mbar_init(bar_s_full0 + 8 * x, 1);
      mbar_init(bar_p_full0 + 8 * x, 4);  // the 4 softmax warps of tile x
      mbar_init(bar_p_free0 + 8 * x, 1);
      mbar_init(bar_o_full0 + 8 * x, 1);
    } else if (lane >= 20 && lane < 20 + kUnitQ) {
      const int k = lane - 20;
      mbar_init(bar_uq_full0 + 8 * k, 1);
      mbar_init(bar_uq_empty0 + 8 * k, kUnitQReaders);
    } else if (lane == 30) {
      mbar_init(smem_addr(&ctl.drain[0]), 1);
      mbar_init(smem_addr(&ctl.drain[1]), 1);
      mbar_init(smem_addr(&ctl.qk_issued_a), 1);
    } else if (lane == 31) {
      mbar_init(bar_q_full, 1);
      mbar_init(bar_q_empty, 1);
      ctl.abort_flag = 0;
    }
    fence_barrier_init();
  }
  if (warp == kWarpQK) {
    tmem_alloc(smem_addr(&ctl.tmem_base), 512);
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
  const int t_end = (p.total_units + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x) *
                    static_cast<int>(gridDim.x);

  if (warp >= kSoftmaxWarps) {
    regs_decrease<kRegsOther>();
    if (warp == kWarpLoad) {
      // ------------------------------------------ TMA: units, Q pairs, K/V
      if (lane == 0) {
        const uint64_t pol_keep = l2_policy_evict_last();   // K/V: re-read by the head's other units
        const uint64_t pol_once = l2_policy_evict_first();  // Q: read once
        uint32_t pos = 0, qcount = 0, kq = 0;               // pos: ring positions filled (K_t at 2t, V_t at 2t+1)
        int t_static = blockIdx.x;
        int t_sched = 0;  // static deal: next unit of the order to look at
        bool ok = true;
        while (ok) {
          int unit = -1;
          UnitPair u;
          for (;;) {
            int cand;
            if (PACKED && p.sched != nullptr) {
              // claimed from the launch's counter (packed batches with a
              // caller-owned counter): any block takes the next unit
              cand = static_cast<int>(atomicAdd(p.sched, 1u));
              if (cand >= p.total_units) break;
            } else if (CAUSAL && sched.n > 0) {
              // the next unit this block owns in the host's deal
              while (t_sched < sched.n &&
                     ((sched.owner[t_sched >> 2] >> (8 * (t_sched & 3))) & 0xffu) != blockIdx.x)
                ++t_sched;
              if (t_sched >= sched.n) break;
              cand = t_sched++;
            } else {
              if (t_static >= t_end) break;
              cand = unit_at<CAUSAL>(p, t_static);
              t_static += gridDim.x;
            }
            if (cand >= p.total_units) continue;
            u = decode_pair<CAUSAL, PACKED>(p, cand);
            if (u.rows[0] > 0) {
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
          if (u.n_max == 0) continue;
          if (!wait_phase(bar_q_empty, (qcount & 1u) ^ 1u, abort_flag, kSiteQEmpty, limit)) { ok = false; break; }
          // both Q tiles (rows past Sq read as zeros and count as loaded)
          mbar_arrive_expect_tx(bar_q_full, 2 * G::kTileBytes);
          for (int x = 0; x < 2; ++x)
            for (int c = 0; c < G::kChunks; ++c) {
              if constexpr (PACKED)  // packed maps are (D, H, tokens, 1)
                tma_load_4d_hint(base + G::kOffQ + x * G::kTileBytes + c * G::kChunkBytes, &map_q, bar_q_full,
                                 c * G::kChunkElems, u.h, u.q_tok0 + kBQ * x, 0, pol_once);
              else                   // padded maps are (D, S, H, B)
                tma_load_4d_hint(base + G::kOffQ + x * G::kTileBytes + c * G::kChunkBytes, &map_q, bar_q_full,
                                 c * G::kChunkElems, u.q0 + kBQ * x, u.h, u.b, pol_once);
            }
          ++qcount;
          for (int j = 0; ok && j < u.n_max; ++j) {
            // paged keys: the cache rows of the tile's two 64-key halves (a
            // half wholly past the sequence's keys reads one row past the end
            // of the cache: zeros)
            int page_tok[2] = {0, 0};
            if constexpr (PACKED) {
              page_tok[0] = page_tok[1] = p.cache_tokens;
            }
            if (PACKED && p.block_table != nullptr) {
              int pg[2] = {0, 0};
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
                const int pos = j * kBK + 64 * hf;
                if (pos < u.kv) pg[hf] = __ldg(p.block_table + static_cast<size_t>(u.b) * p.max_pages + pos / p.page_size);
              }
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
                const int pos = j * kBK + 64 * hf;
                if (pos < u.kv) page_tok[hf] = min(max(pg[hf], 0), p.num_pages - 1) * p.page_size + pos % p.page_size;
              }
            }
            for (int sel = 0; sel < 2; ++sel) {  // K_j, then V_j
              const typename G::Fill f = G::fill_of(pos >> 1, sel != 0);
              if (!wait_phase(bar_kv_empty0 + 8 * f.slot, (f.empty_use & 1u) ^ 1u, abort_flag, kSiteKvEmpty,
                              limit)) {
                ok = false;
                break;
              }
              // (self test only: block 0 leaves out one K fill; the position
              // still counts, so its consumer waits for it in vain)
              if (!(sel == 0 && blockIdx.x == 0 && static_cast<int>(pos >> 1) == p.selftest_skip_fill)) {
                const uint32_t full = (sel ? bar_v_full0 : bar_k_full0) + 8 * f.slot;
                mbar_arrive_expect_tx(full, G::kTileBytes);
                const CUtensorMap* m = sel ? &map_v : &map_k;
                const uint32_t dst = base + G::kOffRing + f.slot * G::kTileBytes;
                if (FP8 && sel && !p.v_rows) {
                  // E4M3 V given transposed, (Sk, D, H, B): the tile is D rows,
                  // each 128 keys long (K-major for the P V product)
                  tma_load_4d_hint(dst, m, full, j * kBK, 0, u.h, u.b, pol_keep);
                } else if (PACKED && p.block_table != nullptr) {
                  // paged: two 64-key boxes, each inside one page (page_size is
                  // a multiple of 64), landing as the two halves of the tile
                  for (int hf = 0; hf < 2; ++hf)
                    for (int c = 0; c < G::kChunks; ++c)
                      tma_load_4d_hint(dst + c * G::kChunkBytes + hf * (G::kChunkBytes / 2), m, full, c * 64, u.h,
                                       page_tok[hf], 0, pol_keep);
                } else if constexpr (PACKED) {
                  for (int c = 0; c < G::kChunks; ++c)
                    tma_load_4d_hint(dst + c * G::kChunkBytes, m, full, c * G::kChunkElems, u.h,
                                     u.k_tok0 + j * kBK, 0, pol_keep);
                } else {
                  for (int c = 0; c < G::kChunks; ++c)
                    tma_load_4d_hint(dst + c * G::kChunkBytes, m, full, c * G::kChunkElems, j * kBK, u.h, u.b,
                                     pol_keep);
                }
              }
              ++pos;
            }
          }
        }
        // Dynamic claims: this block makes no more.  The last block to get
        // here (every block does, aborting or not) puts the counter back to 0
        // for the next launch that uses it.
        if (PACKED && p.sched != nullptr) {
          __threadfence();
          if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
            atomicExch(p.sched, 0u);
            atomicExch(p.sched + 1, 0u);
          }
        }
        // Drains: after a failure every issued copy must land; in any case the
        // issuers' last commit arrivals on the empty barriers must have landed
        // before the block's shared memory is gone.
        if (!ok && qcount > 0) wait_phase_drain(bar_q_full, (qcount - 1) & 1u);
        if (qcount > 0) wait_phase_drain(bar_q_empty, (qcount - 1) & 1u);
        const uint32_t ring = pos;  // positions 0 .. pos - 1 were filled, in order
        for (uint32_t s = 0; s < static_cast<uint32_t>(G::kSlots) && s < ring; ++s) {
          const uint32_t last = ring - 1 - ((ring - 1 - s) % G::kSlots);
          const typename G::Fill f = G::fill_of(last >> 1, (last & 1u) != 0);
          if (!ok) wait_phase_drain(((last & 1u) ? bar_v_full0 : bar_k_full0) + 8 * s, f.full_use & 1u);
          wait_phase_drain(bar_kv_empty0 + 8 * s, f.empty_use & 1u);
        }
      }
      __syncwarp();
    } else if (warp == kWarpQK) {
      // ---------------------------------------------- S_x = Q_x K^T issuer
      uint32_t qcount = 0, tiles = 0, kq = 0;
      uint32_t sc[2] = {0u, 0u};  // S_x products issued
      bool ok = true;
      while (ok) {
        const int unit = take_unit(kq, unit_q, bar_uq_full0, bar_uq_empty0, abort_flag, limit, lane);
        if (unit == -2) { ok = false; break; }
        if (unit < 0) break;
        const UnitPair u = decode_pair<CAUSAL, PACKED>(p, unit);
        if (u.n_max == 0) continue;
        if (!wait_warp(bar_q_full, qcount & 1u, abort_flag, kSiteQFull, limit)) { ok = false; break; }
        ++qcount;
        for (int j = 0; ok && j < u.n_max; ++j, ++tiles) {
          const typename G::Fill f = G::fill_of(tiles, false);
          if (!wait_warp(bar_k_full0 + 8 * f.slot, f.full_use & 1u, abort_flag, kSiteKvFull, limit)) {
            ok = false;
            break;
          }
          const uint32_t ka = base + G::kOffRing + f.slot * G::kTileBytes;
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (j >= u.n[x]) continue;
            // S_x (and the P_x over it) is free once the P V of its previous
            // tile has completed
            if (sc[x] > 0 &&
                !wait_warp(bar_p_free0 + 8 * x, (sc[x] - 1) & 1u, abort_flag, kSitePFree, limit)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t qa = base + G::kOffQ + x * G::kTileBytes;
#pragma unroll
            for (int kk = 0; kk < G::kKSteps; ++kk) {
              const uint32_t off = (kk >> 2) * G::kChunkBytes + (kk & 3) * 32;
              const uint64_t qdesc = sdesc_sw(qa + off, 16, G::kSbo, G::kSwMode);
              const uint64_t kdesc = sdesc_sw(ka + off, 16, G::kSbo, G::kSwMode);
              if constexpr (FP8)
                mma_ss_f8_elect(tmem + G::kTmemS + 128u * x, qdesc, kdesc, p.idesc_qk, kk > 0 ? 1u : 0u);
              else
                mma_ss_elect(tmem + G::kTmemS + 128u * x, qdesc, kdesc, p.idesc_qk, kk > 0 ? 1u : 0u);
            }
            mma_commit_elect(bar_s_full0 + 8 * x);
            if (x == 0) {  // a plain arrive right after the issue
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_addr(&ctl.qk_issued_a));
            }
            ++sc[x];
          }
          if (!ok) break;
          mma_commit_elect(bar_kv_empty0 + 8 * f.slot);
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
      // ---------------------------------------------- O_x += P_x V issuer
      uint32_t tiles = 0, kq = 0;
      uint32_t pc[2] = {0u, 0u};  // P_x V products issued
      bool ok = true;
      while (ok) {
        const int unit = take_unit(kq, unit_q, bar_uq_full0, bar_uq_empty0, abort_flag, limit, lane);
        if (unit == -2) { ok = false; break; }
        if (unit < 0) break;
        const UnitPair u = decode_pair<CAUSAL, PACKED>(p, unit);
        if (u.n_max == 0) continue;
        for (int j = 0; ok && j < u.n_max; ++j, ++tiles) {
          const typename G::Fill f = G::fill_of(tiles, true);
          bool v_ready = false;
          const uint32_t va = base + G::kOffRing + f.slot * G::kTileBytes;
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (j >= u.n[x]) continue;
            if (!wait_warp(bar_p_full0 + 8 * x, pc[x] & 1u, abort_flag, kSitePFull, limit)) {
              ok = false;
              break;
            }
            // P_B V_j goes into the tensor pipe's (in-order) queue after
            // S_A = Q_A K_{j+1}^T, which waits for P_A V_j to complete: queued
            // the other way round, every tile of A would wait for both P V
            // products before its next S.  (pc[0] = index of that S_A product.)
            if (x == 1 && j + 1 < u.n[0] &&
                !wait_warp(smem_addr(&ctl.qk_issued_a), pc[0] & 1u, abort_flag, kSitePvIssued, limit)) {
              ok = false;
              break;
            }
            if (!v_ready) {
              if (!wait_warp(bar_v_full0 + 8 * f.slot, f.full_use & 1u, abort_flag, kSiteKvFull, limit)) {
                ok = false;
                break;
              }
              v_ready = true;
            }
            tc_fence_after_sync();
            // O_x += P_x V_j: P from TMEM (16 keys = 8 columns per MMA), V
            // MN-major in shared memory (LBO = distance between 64-column
            // chunks of D, SBO = 8 keys x 128 B)
            const uint32_t tO = tmem + G::kTmemO + static_cast<uint32_t>(D) * x;
            const uint32_t tP = tmem + G::kTmemS + 128u * x;
            if constexpr (FP8) {
              // E4M3 P (32 keys = 8 columns per MMA, four per column).  V
              // transposed: K-major (D rows of 128 keys, 128-byte swizzle), 32
              // keys = 32 bytes along each row per MMA.  V in rows: MN-major
              // (rows of keys, D contiguous: one swizzle atom wide), 32 keys =
              // 32 rows per MMA.
#pragma unroll
              for (int kk = 0; kk < kBK / 32; ++kk) {
                const uint64_t vdesc = p.v_rows ? sdesc_sw(va + kk * 32 * G::kRowBytes, 16, G::kSbo, G::kSwMode)
                                                : sdesc_sw(va + kk * 32, 16, 1024, kSmemSwizzle128B);
                mma_ts_f8_elect(tO, tP + 8u * kk, vdesc, p.idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < kBK / 16; ++kk)
                mma_ts_elect(tO, tP + 8u * kk, sdesc_sw128(va + kk * 16 * 128, G::kChunkBytes, 1024), p.idesc_pv,
                             (j > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit_elect(bar_p_free0 + 8 * x);
            ++pc[x];
            if (j == u.n[x] - 1) mma_commit_elect(bar_o_full0 + 8 * x);
          }
          if (!ok) break;
          mma_commit_elect(bar_kv_empty0 + 8 * f.slot);
        }
      }
      if (!ok) {
        const uint32_t bar_d = smem_addr(&ctl.drain[1]);
        mma_commit_elect(bar_d);
        wait_phase_drain(bar_d, 0);
      }
    }
  } else {
    regs_increase<kRegsSoftmax>();
    // ---------------------------------------------------------- softmax
    // Thread = one row of tile x; its reference max and sum stay in the
    // thread.  A tile is first exponentiated against the current reference;
    // a row sum above 2^16 (or not a number) shows that some score grew past
    // the reference by more than 16 (log2 units): only then is the exact max
    // taken (the scores reloaded), and if it grew by more than 16 the
    // reference moves and O and the sum are rescaled by 2^(m_old - m_new)
    // (lazy correction, as attn_fwd_kernel's).
    const int x = warp >> 2;
    const int r = threadIdx.x & (kBQ - 1);
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c = p.c;
    const uint32_t tS = tmem + lane_off + G::kTmemS + 128u * x;
    const uint32_t tO = tmem + lane_off + G::kTmemO + static_cast<uint32_t>(D) * x;
    const uint32_t bar_s_full = bar_s_full0 + 8 * x;
    const uint32_t bar_p_full = bar_p_full0 + 8 * x;
    const uint32_t bar_o_full = bar_o_full0 + 8 * x;
    uint32_t sc = 0, oc = 0, kq = 0;
    bool ok = true;
    while (ok) {
      const int unit = take_unit(kq, unit_q, bar_uq_full0, bar_uq_empty0, abort_flag, limit, lane);
      if (unit == -2) { ok = false; break; }
      if (unit < 0) break;
      const UnitPair u = decode_pair<CAUSAL, PACKED>(p, unit);
      const int rows = x ? u.rows[1] : u.rows[0];  // (constant indices keep the unit in registers)
      const int nx = x ? u.n[1] : u.n[0];
      if (rows == 0) continue;  // tile B past the end of the sequence
      const int q0x = u.q0 + kBQ * x;
      const int row = q0x + r;
      const bool row_ok = r < rows;
      size_t row_index, lse_index;  // row of O (in units of D elements) and index into lse
      if constexpr (PACKED) {       // packed: o [total_q, H, D], lse [H, total_q]
        const size_t tok = static_cast<size_t>(u.q_tok0) + kBQ * x + r;
        row_index = tok * p.H + u.h;
        lse_index = static_cast<size_t>(u.h) * p.total_q + tok;
      } else {                      // padded: o [B, H, Sq, D], lse [B, H, Sq]
        row_index = (static_cast<size_t>(u.b) * p.H + u.h) * static_cast<size_t>(p.Sq) + row;
        lse_index = row_index;
      }
      uint16_t* o_dst = p.o + row_index * D;
      if (nx == 0) {  // no valid key for any row of this tile: O = 0, LSE = -inf
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(o_dst);
#pragma unroll
          for (int q = 0; q < D / 8; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
          p.lse[lse_index] = -INFINITY;
        }
        continue;
      }
      float m_used = -INFINITY;  // reference max (log2 units, scale folded in)
      float l = 0.0f;            // sum of 2^(x - m_used) over the row
      bool failed = false;
      for (int j = 0; j < nx; ++j, ++sc) {
        const int k0 = j * kBK;
        const bool masked = (k0 + kBK > u.kv) || (CAUSAL && k0 + kBK - 1 > q0x);
        int climit = u.kv - k0;  // columns >= climit are masked for this row
        if (CAUSAL) climit = min(climit, row - k0 + 1);
        // (a failed wait is warp-uniform and means the block is aborting)
        if (!wait_warp(bar_s_full, sc & 1u, abort_flag, kSiteSFull, limit)) {
          failed = true;
          break;
        }
        tc_fence_after_sync();
        uint32_t sp[128];
        load_s128(tS, sp);
        float sum = 0.0f;
        bool suspect = true;  // the first tile always takes its exact max
        if (j > 0) {
          // each term 2^(x - m_used + shift); partial sums <= 2^(tau + shift)
          // prove that no score of the row grew past the reference by more
          // than tau (the test is also false for NaN / inf)
          float part_max;
          sum = masked ? row_exp128<true, FP8>(sp, c, m_used - PR::kShift, climit, part_max)
                       : row_exp128<false, FP8>(sp, c, m_used - PR::kShift, climit, part_max);
          suspect = !(part_max <= PR::kSumLimit);
        }
        // (warp-uniform decisions: the TMEM loads and stores below are
        // warp-wide instructions)
        if (__any_sync(0xffffffffu, suspect)) {
          if (j > 0) load_s128(tS, sp);  // the raw scores again (P is not stored yet)
          const float mx = masked ? row_max128<true>(sp, climit) : row_max128<false>(sp, climit);
          const float m_tile = (mx == -INFINITY) ? -INFINITY : mx * c;
          bool grow = (j == 0) || m_tile > m_used + PR::kTau;
          float alpha = 1.0f;
          if (grow && j > 0) alpha = ex2_approx(m_used - m_tile);
          if (grow) m_used = m_tile;
          const float mb = (m_used == -INFINITY) ? 0.0f : m_used - PR::kShift;
          float unused;
          sum = masked ? row_exp128<true, FP8>(sp, c, mb, climit, unused)
                       : row_exp128<false, FP8>(sp, c, mb, climit, unused);
          if (j > 0 && __any_sync(0xffffffffu, grow)) {
            // O_x holds the products of the tiles before (all completed: this
            // S_x was written after the last of them): rescale this row
            l *= alpha;
            const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
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
        }
        // P over the first columns of S_x (their scores are in registers):
        // 64 columns of bf16 pairs, or 32 of four E4M3 values
#pragma unroll
        for (int q = 0; q < G::kPCols / 16; ++q)
          tmem_st_32x32b_x16(tS + 16 * q, *reinterpret_cast<const uint32_t(*)[16]>(&sp[16 * q]));
        tmem_st_wait();
        warp_arrive_after_tc(bar_p_full, lane);
        l += sum;
      }
      if (failed) { ok = false; break; }
      // ------------------------------------------------------------ epilogue
      if (!wait_warp(bar_o_full, oc & 1u, abort_flag, kSiteOFull, limit)) { ok = false; break; }
      ++oc;
      tc_fence_after_sync();
      const bool has_key = l > 0.0f;
      const float inv_l = has_key ? p.v_scale * rcp_approx(l) : 0.0f;  // (v_scale: 1, or the E4M3 V descale)
      const float lse_row = has_key ? (m_used - PR::kShift + lg2_approx(l)) * kLn2 : -INFINITY;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tO + q * 32, o);
        tmem_ld_wait_x32(o);
        if (row_ok) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = has_key ? pack_bf16x2(u2f(o[2 * e]) * inv_l, u2f(o[2 * e + 1]) * inv_l) : 0u;
          if (p.o_align32) {
            st_global_v8(o_dst + q * 32, *reinterpret_cast<const uint32_t(*)[8]>(&w[0]));
            st_global_v8(o_dst + q * 32 + 16, *reinterpret_cast<const uint32_t(*)[8]>(&w[8]));
          } else {
            uint4* dst = reinterpret_cast<uint4*>(o_dst + q * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
          }
        }
      }
      // the next unit's first P V overwrites O_x only after this warpgroup's
      // p_full for it, which comes after these loads
      tc_fence_before_sync();
      if (row_ok) p.lse[lse_index] = lse_row;
    }
    // The commit of the last P_x V lands asynchronously and nothing else
    // waits for it: wait before exiting.
    if (sc > 0) wait_phase_drain(bar_p_free0 + 8 * x, (sc - 1) & 1u);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpQK) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// dynamic shared memory attribute set, per device and instantiation
constexpr int kMaxDevicesPair = 64;
std::atomic<bool> g_pair_smem_set[kMaxDevicesPair][12];

// Cost model of a unit, in hundredths of the time one 128-key tile takes the
// one-tile kernel.  Which kernel runs: non-causal, a key tile that both query
// tiles of a pair process costs 184 (measured: 1527 against 1390 TFLOP/s on
// the S = 8192 workload); causal, constants fitted by least squares to the
// launch times of both kernels on causal batches (D = 128, S = 1024 to 8192,
// 128 to 4096 query tiles; within 3 us of every time): a key tile of both
// query tiles 181, the fixed part of a single-tile unit (Q load, first tile,
// epilogue) 298, and the fixed part of a pair together with its last key
// tile, which only tile B processes, 996 (taken as 498 each; the fit cannot
// tell the two apart, as every causal pair has one such tile).  The static
// deal of causal pairs weighs them 184 (both tiles), 130 (tile B alone) and
// 200 (fixed part): dealt with the fitted weights instead, batches of 32 and
// 64 heads at 4096 and 8192 keys ran 1.6 % and 2 % slower.
struct PairWeights {
  int64_t both, alone, unit;
};
constexpr int64_t kCostTile = 100, kCostBothDense = 184, kCostUnit = 298;
// E4M3 or D = 64, non-causal: a key tile of both query tiles costs 170
// (measured on the E4M3 S = 8192 workload: 656 against 773 us at 7 against 14
// waves; bf16 D = 64 S = 1024, 4 against 7 waves: 58 against 66 us): their
// faster products leave the softmax the longer part, which the pair
// interleaves.
constexpr int64_t kCostBothDenseLight = 170;
constexpr PairWeights kRouteWeights{181, 498, 498}, kDealWeights{184, 130, 200};

int64_t key_tiles(int64_t q0, int64_t rows, int64_t Sk, bool causal) {
  if (rows <= 0) return 0;
  const int64_t lim = causal ? std::min(Sk, q0 + rows) : Sk;
  return (lim + kBK - 1) / kBK;
}

// modelled time of single-tile unit `qt` and of pair unit `pr`
int64_t tile_cost(int64_t qt, int64_t Sq, int64_t Sk, bool causal) {
  const int64_t q0 = qt * kBQ;
  return key_tiles(q0, std::min<int64_t>(kBQ, Sq - q0), Sk, causal) * kCostTile + kCostUnit;
}

int64_t pair_cost(int64_t pr, int64_t Sq, int64_t Sk, bool causal, const PairWeights& w) {
  const int64_t q0 = pr * 2 * kBQ;
  const int64_t na = key_tiles(q0, std::min<int64_t>(kBQ, Sq - q0), Sk, causal);
  const int64_t nb = key_tiles(q0 + kBQ, std::min<int64_t>(kBQ, Sq - q0 - kBQ), Sk, causal);
  const int64_t both = std::min(na, nb);
  return both * w.both + (std::max(na, nb) - both) * w.alone + w.unit;
}

struct CachedSchedule {
  int B = -1, H = 0, Sq = 0, Sk = 0, head_group = 0, grid = 0;
  int64_t n = 0;
  uint8_t owner[kSchedMaxUnits];
};
constexpr int kScheduleCacheSize = 8;
std::mutex g_sched_mutex;
CachedSchedule g_sched_cache[kScheduleCacheSize];
int g_sched_next = 0;

// The schedule for a causal launch, built once per shape and kept in a small
// cache (the deal of up to 4096 units costs tens of microseconds of host time).
bool causal_schedule(const Params& p, int grid, UnitSched<true>& out) {
  std::lock_guard<std::mutex> lock(g_sched_mutex);
  CachedSchedule* hit = nullptr;
  for (CachedSchedule& c : g_sched_cache)
    if (c.B == p.B && c.H == p.H && c.Sq == p.Sq && c.Sk == p.Sk && c.head_group == p.head_group && c.grid == grid)
      hit = &c;
  if (hit == nullptr) {
    CachedSchedule& c = g_sched_cache[g_sched_next];
    c.B = -1;
    c.n = attn_pair_host::build_schedule(p.B, p.H, p.Sq, p.Sk, p.head_group, grid, c.owner, kSchedMaxUnits);
    if (c.n < 0) return false;
    c.B = p.B;
    c.H = p.H;
    c.Sq = p.Sq;
    c.Sk = p.Sk;
    c.head_group = p.head_group;
    c.grid = grid;
    g_sched_next = (g_sched_next + 1) % kScheduleCacheSize;
    hit = &c;
  }
  out.n = static_cast<int>(hit->n);
  std::memset(out.owner, 0, sizeof(out.owner));
  std::memcpy(out.owner, hit->owner, static_cast<size_t>(hit->n));  // little-endian bytes: entry t is byte t
  return true;
}

template <int D, bool CAUSAL, bool FP8, bool PACKED = false>
attn_status launch_pair(int dev, int num_sms, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                        const Params& p0, cudaStream_t stream) {
  static_assert(!(FP8 && PACKED), "packed batches are bf16");
  auto kern = attn_fwd_pair_kernel<D, CAUSAL, FP8, PACKED>;
  constexpr int smem = GeoPair<D, FP8>::kSmemBytes;
  constexpr int idx = PACKED ? 8 + (D == 64 ? 0 : 2) + (CAUSAL ? 1 : 0)
                             : (D == 64 ? 0 : 4) + (CAUSAL ? 2 : 0) + (FP8 ? 1 : 0);
  if (dev < 0 || dev >= kMaxDevicesPair) return ATTN_ERR_UNSUPPORTED_DEVICE;
  if (!g_pair_smem_set[dev][idx].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return ATTN_ERR_CUDA;
    g_pair_smem_set[dev][idx].store(true, std::memory_order_release);
  }
  const int grid = p0.total_units < num_sms ? p0.total_units : num_sms;
  UnitSched<CAUSAL> sched;
  sched.n = 0;
  if constexpr (CAUSAL) {
    // padded batches only: a packed batch's sequence lengths are on the
    // device, so its units keep the round-robin deal
    if (PACKED || !causal_schedule(p0, grid, sched)) sched.n = 0;
  }
  kern<<<grid, kThreads, smem, stream>>>(mq, mk, mv, with_divisors(p0, grid), sched);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

namespace attn_pair_host {

bool use_pair(int B, int H, int Sq, int Sk, int D, bool causal, int num_sms, bool fp8) {
  if (B <= 0 || H <= 0 || Sq <= kBQ || Sk < 0 || num_sms < 1 || (D != 64 && D != 128)) return false;
  // E4M3 or D = 64: products that take half the bf16 D = 128 time (or less),
  // so the softmax, which the pair interleaves, weighs more
  const bool light = fp8 || D == 64;
  const int64_t bh = static_cast<int64_t>(B) * H;
  const int64_t g = num_sms;
  const int64_t n_tiles = (static_cast<int64_t>(Sq) + kBQ - 1) / kBQ;
  const int64_t n_pairs = (static_cast<int64_t>(Sq) + 2 * kBQ - 1) / (2 * kBQ);
  if (!causal) {
    // units of one length: waves of units over the SMs
    const int64_t both = light ? kCostBothDenseLight : kCostBothDense;
    return both * ((bh * n_pairs + g - 1) / g) < kCostTile * ((bh * n_tiles + g - 1) / g);
  }
  // causal units of many lengths, dealt longest first: the time is about the
  // larger of the longest unit and the mean work per SM; the pair kernel
  // needs its static deal (at most 4096 units) to balance
  if (bh * n_pairs > kSchedMaxUnits) return false;
  // light products from 1024 (E4M3) or 2048 (bf16 D = 64) queries on: the
  // pair measured faster on every such causal batch timed (E4M3 S = 1024 to
  // 8192: 4-26 %; D = 64 S = 2048 to 8192: 6-24 %, but 4 % slower at 1024);
  // shorter ones take the model
  if (light && Sq >= (fp8 ? 1024 : 2048)) return true;
  int64_t one_total = 0, one_max = 0, pair_total = 0, pair_max = 0;
  for (int64_t t = 0; t < n_tiles; ++t) {
    const int64_t c = tile_cost(t, Sq, Sk, true);
    one_total += c;
    one_max = std::max(one_max, c);
  }
  for (int64_t t = 0; t < n_pairs; ++t) {
    const int64_t c = pair_cost(t, Sq, Sk, true, kRouteWeights);
    pair_total += c;
    pair_max = std::max(pair_max, c);
  }
  const int64_t one = std::max(one_max, (bh * one_total + g - 1) / g);
  const int64_t pair = std::max(pair_max, (bh * pair_total + g - 1) / g);
  return pair < one;
}

int64_t build_schedule(int B, int H, int Sq, int Sk, int head_group, int grid, uint8_t* owner, int64_t max_units) {
  if (B < 0 || H < 0 || Sq < 0 || Sk < 0 || head_group < 1 || grid < 1 || grid > 256 || owner == nullptr)
    return -1;
  const int64_t bh = static_cast<int64_t>(B) * H;
  const int64_t n_pairs = (static_cast<int64_t>(Sq) + 2 * kBQ - 1) / (2 * kBQ);
  const int64_t n = bh * n_pairs;
  if (n > max_units) return -1;
  // the kernel's unit order (decode_pair<true>): groups of head_group heads,
  // within a group the pairs from the last one down, each over the group's heads
  using Load = std::pair<int64_t, int>;
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> free_at;
  for (int b = 0; b < grid; ++b) free_at.push({0, b});
  int64_t t = 0;
  for (int64_t g0 = 0; g0 < bh; g0 += head_group) {
    const int64_t heads = std::min<int64_t>(head_group, bh - g0);
    for (int64_t wq = 0; wq < n_pairs; ++wq) {
      const int64_t c = pair_cost(n_pairs - 1 - wq, Sq, Sk, true, kDealWeights);
      for (int64_t h = 0; h < heads; ++h, ++t) {
        const Load l = free_at.top();
        free_at.pop();
        owner[t] = static_cast<uint8_t>(l.second);
        free_at.push({l.first + c, l.second});
      }
    }
  }
  return n;
}

attn_status launch(int D, bool causal, bool fp8, int num_sms, const CUtensorMap& mq, const CUtensorMap& mk,
                   const CUtensorMap& mv, const attn_detail::Params& p, cudaStream_t s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (p.cu_q != nullptr) {  // packed or paged (bf16)
    if (fp8) return ATTN_ERR_SHAPE;
    if (causal)
      return D == 64 ? launch_pair<64, true, false, true>(dev, num_sms, mq, mk, mv, p, s)
                     : launch_pair<128, true, false, true>(dev, num_sms, mq, mk, mv, p, s);
    return D == 64 ? launch_pair<64, false, false, true>(dev, num_sms, mq, mk, mv, p, s)
                   : launch_pair<128, false, false, true>(dev, num_sms, mq, mk, mv, p, s);
  }
  if (fp8) {
    if (causal)
      return D == 64 ? launch_pair<64, true, true>(dev, num_sms, mq, mk, mv, p, s)
                     : launch_pair<128, true, true>(dev, num_sms, mq, mk, mv, p, s);
    return D == 64 ? launch_pair<64, false, true>(dev, num_sms, mq, mk, mv, p, s)
                   : launch_pair<128, false, true>(dev, num_sms, mq, mk, mv, p, s);
  }
  if (causal)
    return D == 64 ? launch_pair<64, true, false>(dev, num_sms, mq, mk, mv, p, s)
                   : launch_pair<128, true, false>(dev, num_sms, mq, mk, mv, p, s);
  return D == 64 ? launch_pair<64, false, false>(dev, num_sms, mq, mk, mv, p, s)
                 : launch_pair<128, false, false>(dev, num_sms, mq, mk, mv, p, s);
}

attn_status status_read_clear(uint32_t host[3]) {
  host[0] = host[1] = host[2] = 0;
  if (cudaMemcpyFromSymbol(host, g_attn_status, 3 * sizeof(uint32_t)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (host[0] == 0) return ATTN_OK;
  const uint32_t zero[3] = {0, 0, 0};
  if (cudaMemcpyToSymbol(g_attn_status, zero, sizeof(zero)) != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // namespace attn_pair_host
