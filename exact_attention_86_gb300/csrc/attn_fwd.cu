// Exact fused attention forward for GB300 (sm_103a).
//
// Computes O = softmax(scale * Q K^T + mask) V and LSE = ln(sum_j exp(scale * q.k_j))
// for a padded batch [B, H, S, D] of bf16 tensors ("Kernel Fusion and the Memory
// Wall", section "FlashAttention: avoid the full score matrix").  Each CTA owns a
// block of 2 x 128 query rows at a time and streams the K/V tiles of that head
// past them ("Attention softmax fusion", section "The tile loop"); the score
// tile lives only in Tensor Memory and registers, and the running max / sum /
// numerator are corrected by exp(m_old - m_new) whenever a later tile raises the
// row maximum (same section, second paragraph).  Nothing of size Sq x Sk is ever
// written to device memory.
//
// CTA layout (384 threads, persistent over work units):
//   warps 0-3  softmax warpgroup 0: rows 0-127 of the unit (one thread per row)
//   warps 4-7  softmax warpgroup 1: rows 128-255
//   warp 8     TMA producer (one elected lane)
//   warp 9     TMEM owner and tcgen05.mma issuer (one elected lane)
//   warps 10-11 idle (they complete warpgroup 2 for the register split)
// The block launches with 168 registers per thread; warpgroup 2 gives registers
// back (120 each) and the softmax warpgroups take 192 each, so a whole
// 128-column score row stays in registers without spills:
//   launch 384 x 168 = 64512 = 256 x 192 + 128 x 120;
//   per SM sub-partition (one warp of each warpgroup): (192+192+120) x 32 <= 16384.
//
// Tensor Memory (512 columns x 128 lanes, fp32):
//   [  0,128)  S0: scores of Q tile 0 vs the current K tile; its first 64
//              columns are overwritten by P0 (bf16 pairs) once softmax is done
//   [128,256)  S1 / P1 for Q tile 1
//   [256,256+D)     O0 accumulator,  [256+D,256+2D) O1 accumulator
//
// Per K/V tile j the MMA lane issues, in this order,
//   O0 += P0(j) V_j ; S0 = Q0 K_{j+1}^T ; O1 += P1(j) V_j ; S1 = Q1 K_{j+1}^T
// so that softmax of one Q tile overlaps the tensor-core work of the other.
// tcgen05.mma operations issued by one thread execute in order, so the QK^T of
// tile j+1 may overwrite the columns that the preceding PV of tile j reads.
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
#include <mutex>

#include "attn.h"
#include "sm103_ptx.cuh"

using namespace attn_sm103;

namespace {

constexpr int kBQ = 128;          // query rows per Q tile (MMA M, TMEM lanes)
constexpr int kBK = 128;          // keys per K/V tile (MMA N of QK^T)
constexpr int kQT = 2;            // Q tiles per work unit, sharing each K/V tile
constexpr int kUnitRows = kQT * kBQ;
constexpr int kThreads = 384;
constexpr int kRegsSoftmax = 192;
constexpr int kRegsOther = 120;
constexpr int kWarpLoad = 8;
constexpr int kWarpMma = 9;
constexpr float kTau = 8.0f;      // lazy rescale threshold (log2 units)
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
};

// [0]: 1 once any wait gave up; [1]: site of the first one; [2]: its block.
__device__ uint32_t g_attn_status[3];

template <int D>
struct Geo {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kTileBytes = 128 * D * 2;     // one Q, K or V tile (128 rows)
  static constexpr int kChunkBytes = 128 * 128;      // 128 rows x 64 bf16 (one 128-B swizzle column)
  static constexpr int kChunks = D / 64;
  static constexpr int kSlots = (D == 128) ? 4 : 8;  // K/V ring depth (tiles)
  static __host__ __device__ constexpr uint32_t tmem_s(int i) { return 128u * i; }
  static __host__ __device__ constexpr uint32_t tmem_o(int i) { return 256u + D * i; }
  static constexpr int kTmemCols = 512;
  static constexpr int kOffQ = 1024;                 // after the control block
  static constexpr int kOffRing = kOffQ + kQT * kTileBytes;
  static constexpr int kSmemBytes = kOffRing + kSlots * kTileBytes + 1024;  // + alignment slack
};

struct Ctrl {
  uint64_t q_full, q_empty;
  uint64_t kv_full[8], kv_empty[8];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Ctrl) <= 1024, "control block");

struct Params {
  uint16_t* o;
  float* lse;
  const int32_t* kv_lens;
  int B, H, Sq, Sk;
  int n_qpairs;
  int total_units;
  float c;                 // |scale| * log2(e)
  uint32_t idesc_qk;       // negate-A set when scale < 0
  uint32_t idesc_pv;
  uint64_t wait_limit_ns;
};

struct Unit {
  int b, h, q0;
  int kv;                  // valid keys of this batch entry (kv_lens clamped to [0, Sk])
  int n[2];                // K tiles each Q tile needs (0: tile absent or no valid key)
};

template <bool CAUSAL>
__device__ __forceinline__ Unit decode_unit(const Params& p, int t) {
  Unit u;
  const int bh_count = p.B * p.H;
  int qp, bh;
  if (CAUSAL) {  // longest units first: query blocks from the end of the sequence
    qp = p.n_qpairs - 1 - t / bh_count;
    bh = t % bh_count;
  } else {       // consecutive units share a head, so its K/V stay hot in L2
    qp = t % p.n_qpairs;
    bh = t / p.n_qpairs;
  }
  u.b = bh / p.H;
  u.h = bh % p.H;
  u.q0 = qp * kUnitRows;
  int kv = p.Sk;
  if (p.kv_lens != nullptr) kv = min(max(__ldg(p.kv_lens + u.b), 0), p.Sk);
  u.kv = kv;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r_first = u.q0 + i * kBQ;
    if (r_first >= p.Sq) {
      u.n[i] = 0;
    } else {
      int lim = kv;
      if (CAUSAL) lim = min(lim, min(r_first + kBQ, p.Sq));  // last row of the tile + 1
      u.n[i] = (lim + kBK - 1) / kBK;
    }
  }
  return u;
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

// Wait used only while draining after an abort: ignores the abort flag.
__device__ __forceinline__ void wait_phase_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kDrainLimitNs) return;
  }
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const Params p) {
  using G = Geo<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  Ctrl& ctl = *reinterpret_cast<Ctrl*>(smem_raw + (base - raw));
  volatile int* abort_flag = &ctl.abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const uint32_t bar_q_full = smem_addr(&ctl.q_full);
  const uint32_t bar_q_empty = smem_addr(&ctl.q_empty);
  const uint32_t bar_kv_full0 = smem_addr(&ctl.kv_full[0]);
  const uint32_t bar_kv_empty0 = smem_addr(&ctl.kv_empty[0]);
  const uint32_t bar_drain = smem_addr(&ctl.drain);

  if (threadIdx.x == 0) {
    mbar_init(bar_q_full, 1);
    mbar_init(bar_q_empty, 1);
    for (int s = 0; s < G::kSlots; ++s) {
      mbar_init(bar_kv_full0 + 8 * s, 1);
      mbar_init(bar_kv_empty0 + 8 * s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&ctl.s_full[i]), 1);
      mbar_init(smem_addr(&ctl.p_full[i]), kBQ);
      mbar_init(smem_addr(&ctl.o_full[i]), 1);
    }
    mbar_init(bar_drain, 1);
    ctl.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMma) {
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

  if (warp >= 8) {
    // ------------------------------------------- warpgroup 2: TMA and MMA
    regs_decrease<kRegsOther>();
  if (warp == kWarpLoad) {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      const uint64_t pol_keep = l2_policy_evict_last();   // K/V: re-read by every query block of the head
      const uint64_t pol_once = l2_policy_evict_first();  // Q: read once
      uint32_t ring = 0, qcount = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.total_units; t += gridDim.x) {
        const Unit u = decode_unit<CAUSAL>(p, t);
        const int N = max(u.n[0], u.n[1]);
        if (N == 0) continue;
        if (!wait_phase(bar_q_empty, (qcount & 1u) ^ 1u, abort_flag, kSiteQEmpty, limit)) { ok = false; break; }
        mbar_arrive_expect_tx(bar_q_full, (u.n[0] > 0 ? G::kTileBytes : 0) + (u.n[1] > 0 ? G::kTileBytes : 0));
        for (int i = 0; i < 2; ++i) {
          if (u.n[i] == 0) continue;
          for (int c = 0; c < G::kChunks; ++c)
            tma_load_4d_hint(base + G::kOffQ + i * G::kTileBytes + c * G::kChunkBytes, &map_q, bar_q_full, c * 64,
                             u.q0 + i * kBQ, u.h, u.b, pol_once);
        }
        ++qcount;
        for (int j = 0; ok && j < N; ++j) {
          for (int sel = 0; sel < 2; ++sel) {  // K_j, then V_j
            const uint32_t slot = ring % G::kSlots;
            const uint32_t ph = (ring / G::kSlots) & 1u;
            if (!wait_phase(bar_kv_empty0 + 8 * slot, ph ^ 1u, abort_flag, kSiteKvEmpty, limit)) { ok = false; break; }
            const uint32_t full = bar_kv_full0 + 8 * slot;
            mbar_arrive_expect_tx(full, G::kTileBytes);
            const CUtensorMap* m = sel ? &map_v : &map_k;
            for (int c = 0; c < G::kChunks; ++c)
              tma_load_4d_hint(base + G::kOffRing + slot * G::kTileBytes + c * G::kChunkBytes, m, full, c * 64,
                               j * kBK, u.h, u.b, pol_keep);
            ++ring;
          }
        }
      }
      if (!ok) {
        // Let every copy this lane started land before the CTA exits.
        if (qcount > 0) wait_phase_drain(bar_q_full, (qcount - 1) & 1u);
        for (uint32_t s = 0; s < (uint32_t)G::kSlots && s < ring; ++s) {
          const uint32_t last = ring - 1 - ((ring - 1 - s) % G::kSlots);  // last load issued into slot s
          wait_phase_drain(bar_kv_full0 + 8 * s, (last / G::kSlots) & 1u);
        }
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      uint32_t ring = 0, qcount = 0;
      uint32_t pcount0 = 0u, pcount1 = 0u;
      bool ok = true;
      // barrier of Q tile i = barrier of tile 0 + 8 * i (consecutive uint64_t)
      const uint32_t bar_s_full0 = smem_addr(&ctl.s_full[0]);
      const uint32_t bar_p_full0 = smem_addr(&ctl.p_full[0]);
      const uint32_t bar_o_full0 = smem_addr(&ctl.o_full[0]);

      // S_i = Q_i K^T: both operands K-major, 128-B swizzled; one MMA per 16 columns of D.
      auto issue_qk = [&](int i, uint32_t slot) {
        const uint32_t qa = base + G::kOffQ + i * G::kTileBytes;
        const uint32_t ka = base + G::kOffRing + slot * G::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * G::kChunkBytes + (kk & 3) * 32;
          mma_ss(tmem + G::tmem_s(i), sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024), p.idesc_qk,
                 kk > 0 ? 1u : 0u);
        }
      };
      // O_i += P_i V: P from TMEM (16 keys = 8 columns per MMA), V MN-major in smem
      // (LBO = distance between 64-column chunks of D, SBO = 8 keys x 128 B).
      auto issue_pv = [&](int i, uint32_t slot, bool accumulate) {
        const uint32_t va = base + G::kOffRing + slot * G::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          mma_ts(tmem + G::tmem_o(i), tmem + G::tmem_s(i) + kk * 8,
                 sdesc_sw128(va + kk * 16 * 128, G::kChunkBytes, 1024), p.idesc_pv,
                 (accumulate || kk > 0) ? 1u : 0u);
        }
      };
      auto wait_kv = [&](uint32_t pos) -> bool {
        const uint32_t slot = pos % G::kSlots;
        if (!wait_phase(bar_kv_full0 + 8 * slot, (pos / G::kSlots) & 1u, abort_flag, kSiteKvFull, limit)) return false;
        tc_fence_after_sync();
        return true;
      };

      for (int t = blockIdx.x; ok && t < p.total_units; t += gridDim.x) {
        const Unit u = decode_unit<CAUSAL>(p, t);
        const int N = max(u.n[0], u.n[1]);
        if (N == 0) continue;
        if (!wait_phase(bar_q_full, qcount & 1u, abort_flag, kSiteQFull, limit)) { ok = false; break; }
        ++qcount;
        tc_fence_after_sync();
        if (!wait_kv(ring)) { ok = false; break; }
        for (int i = 0; i < 2; ++i) {
          if (u.n[i] > 0) {
            issue_qk(i, ring % G::kSlots);
            mma_commit(bar_s_full0 + 8 * i);
          }
        }
        mma_commit(bar_kv_empty0 + 8 * (ring % G::kSlots));
        for (int j = 0; ok && j < N; ++j) {
          const uint32_t v_pos = ring + 2 * j + 1;
          const uint32_t kn_pos = ring + 2 * j + 2;
          if (!wait_kv(v_pos)) { ok = false; break; }
          bool kn_ready = false;
          for (int i = 0; i < 2; ++i) {
            if (j >= u.n[i]) continue;
            uint32_t& pc = i ? pcount1 : pcount0;
            if (!wait_phase(bar_p_full0 + 8 * i, pc & 1u, abort_flag, kSitePFull, limit)) { ok = false; break; }
            ++pc;
            tc_fence_after_sync();
            issue_pv(i, v_pos % G::kSlots, j > 0);
            if (j + 1 < u.n[i]) {
              if (!kn_ready) {
                if (!wait_kv(kn_pos)) { ok = false; break; }
                kn_ready = true;
              }
              issue_qk(i, kn_pos % G::kSlots);
              mma_commit(bar_s_full0 + 8 * i);
            } else {
              mma_commit(bar_o_full0 + 8 * i);
            }
          }
          if (!ok) break;
          if (kn_ready) mma_commit(bar_kv_empty0 + 8 * (kn_pos % G::kSlots));
          mma_commit(bar_kv_empty0 + 8 * (v_pos % G::kSlots));
        }
        if (!ok) break;
        ring += 2 * N;
        mma_commit(bar_q_empty);
      }
      if (!ok) {
        // Let every MMA this lane issued retire before TMEM is released.
        mma_commit(bar_drain);
        wait_phase_drain(bar_drain, 0);
      }
    }
    __syncwarp();
  }
  } else {
    // ------------------------------------------- warpgroups 0, 1: softmax
    regs_increase<kRegsSoftmax>();
    const int wg = warp >> 2;                      // which Q tile of the unit
    const int r = threadIdx.x & (kBQ - 1);         // row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + G::tmem_s(wg);
    const uint32_t tO = tmem + lane_off + G::tmem_o(wg);
    const uint32_t bar_s = smem_addr(&ctl.s_full[wg]);
    const uint32_t bar_p = smem_addr(&ctl.p_full[wg]);
    const uint32_t bar_o = smem_addr(&ctl.o_full[wg]);
    const float c = p.c;
    uint32_t scount = 0, ocount = 0;
    bool ok = true;

    for (int t = blockIdx.x; ok && t < p.total_units; t += gridDim.x) {
      const Unit u = decode_unit<CAUSAL>(p, t);
      const int tile_row0 = u.q0 + wg * kBQ;
      if (tile_row0 >= p.Sq) continue;
      const int row = tile_row0 + r;
      const size_t row_index = (static_cast<size_t>(u.b) * p.H + u.h) * static_cast<size_t>(p.Sq) + row;
      const int n = wg ? u.n[1] : u.n[0];
      if (n == 0) {  // no valid key for any row of this tile: O = 0, LSE = -inf
        if (row < p.Sq) {
          uint4* dst = reinterpret_cast<uint4*>(p.o + row_index * D);
#pragma unroll
          for (int q = 0; q < D / 8; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
          p.lse[row_index] = -INFINITY;
        }
        continue;
      }

      float m_used = -INFINITY;  // stale running max (log2 units, scale folded in)
      float l = 0.0f;            // running sum of 2^(x - m_used)
      for (int j = 0; j < n; ++j) {
        if (!wait_phase(bar_s, scount & 1u, abort_flag, kSiteSFull, limit)) { ok = false; break; }
        ++scount;
        tc_fence_after_sync();
        uint32_t s[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld_32x32b_x32(tS + q * 32, s[q]);
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld_wait_x32(s[q]);

        const int k0 = j * kBK;
        const bool masked = (k0 + kBK > u.kv) || (CAUSAL && k0 + kBK - 1 > tile_row0);
        int climit = u.kv - k0;  // columns >= climit are masked for this row
        if (CAUSAL) climit = min(climit, row - k0 + 1);

        // row maximum of the valid raw scores (8 independent chains of 3-input max)
        float mx8[8];
        if (masked) {
#pragma unroll
          for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
#pragma unroll
          for (int col = 0; col < kBK; col += 2) {
            const float x0 = (col < climit) ? u2f(s[col >> 5][col & 31]) : -INFINITY;
            const float x1 = (col + 1 < climit) ? u2f(s[col >> 5][(col + 1) & 31]) : -INFINITY;
            mx8[(col >> 1) & 7] = max3(mx8[(col >> 1) & 7], x0, x1);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) mx8[e] = u2f(s[0][e]);
#pragma unroll
          for (int col = 8; col < kBK; col += 2)
            mx8[(col >> 1) & 7] = max3(mx8[(col >> 1) & 7], u2f(s[col >> 5][col & 31]), u2f(s[col >> 5][(col + 1) & 31]));
        }
        const float mx = max3(max3(mx8[0], mx8[1], mx8[2]), max3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
        const float m_tile = (mx == -INFINITY) ? -INFINITY : mx * c;
        const float m_new = fmaxf(m_used, m_tile);
        // Lazy correction: move the reference max only when it grew by more than
        // kTau; every term stays <= 2^kTau, and O and l keep one shared reference.
        const bool grow = m_new > m_used + kTau;
        const float alpha = grow ? ex2_approx(m_used - m_new) : 1.0f;
        if (grow) {
          l *= alpha;
          m_used = m_new;
        }
        // p = 2^(s*c - mb) on pairs (one packed FMA per pair), packed row sum,
        // bf16 pairs written back over the first half of the S columns in
        // 16-column chunks.
        const float mb = (m_used == -INFINITY) ? 0.0f : m_used;
        const uint64_t c2 = f2_pack(c, c);
        const uint64_t nmb2 = f2_pack(-mb, -mb);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int col = q * 32 + 2 * e;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(u2f(s[q][2 * e]), u2f(s[q][2 * e + 1])), c2, nmb2), x0, x1);
            float p0 = ex2_approx(x0);
            float p1 = ex2_approx(x1);
            if (masked) {
              p0 = (col < climit) ? p0 : 0.0f;
              p1 = (col + 1 < climit) ? p1 : 0.0f;
            }
            acc[e & 3] = f2_add(acc[e & 3], f2_pack(p0, p1));
            pk[e] = pack_bf16x2(p0, p1);
          }
          tmem_st_32x32b_x16(tS + q * 16, pk);
        }
        {
          const uint64_t a01 = f2_add(acc[0], acc[1]);
          const uint64_t a23 = f2_add(acc[2], acc[3]);
          float lo, hi;
          f2_unpack(f2_add(a01, a23), lo, hi);
          l += lo + hi;
        }
        if (j > 0 && __any_sync(0xffffffffu, grow)) {
          // O_i row *= alpha (PV of tile j-1 has retired: S_i(j) was committed after it).
          // Done after P is written so that the score row is no longer live.
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
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(bar_p);
      }
      if (!ok) break;

      // ------------------------------------------------------------ epilogue
      if (!wait_phase(bar_o, ocount & 1u, abort_flag, kSiteOFull, limit)) { ok = false; break; }
      ++ocount;
      tc_fence_after_sync();
      const bool has_key = l > 0.0f;
      const float inv_l = has_key ? 1.0f / l : 0.0f;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tO + q * 32, o);
        tmem_ld_wait_x32(o);
        if (row < p.Sq) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = has_key ? pack_bf16x2(u2f(o[2 * e]) * inv_l, u2f(o[2 * e + 1]) * inv_l) : 0u;
          uint4* dst = reinterpret_cast<uint4*>(p.o + row_index * D + q * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
      }
      if (row < p.Sq) p.lse[row_index] = has_key ? (m_used + log2f(l)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
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

// ------------------------------------------------------------------- host side

struct DeviceInfo {
  int initialised = 0;
  int supported = 0;
  int num_sms = 0;
  bool smem_set[4] = {false, false, false, false};
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

// Rank-4 map over [B, H, S, D] (D innermost) with a 64 x 128 box (one 128-B
// swizzle column of a tile).  Rows past S read as zeros and never spill into the
// next head.
bool make_map(CUtensorMap* m, const void* ptr, int B, int H, int S, int D) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = encoder();
  if (encode == nullptr) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)S * D * 2, (cuuint64_t)H * S * D * 2};
  const cuuint32_t box[4] = {64, 128, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool CAUSAL>
attn_status launch(DeviceInfo& dev, int idx, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                   const Params& p, cudaStream_t stream) {
  auto kern = attn_fwd_kernel<D, CAUSAL>;
  constexpr int smem = Geo<D>::kSmemBytes;
  if (!dev.smem_set[idx]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return ATTN_ERR_CUDA;
    dev.smem_set[idx] = true;
  }
  const int grid = p.total_units < dev.num_sms ? p.total_units : dev.num_sms;
  kern<<<grid, kThreads, smem, stream>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" {

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Sq, int Sk,
                     int D, float scale, int causal, const int32_t* kv_lens, attn_stream_t stream) {
  if (B < 0 || H < 0 || Sq < 0 || Sk < 0) return ATTN_ERR_SHAPE;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED_D;
  if (!std::isfinite(scale)) return ATTN_ERR_SCALE;
  if (B == 0 || H == 0 || Sq == 0) return ATTN_OK;
  if (q == nullptr || o == nullptr || lse == nullptr) return ATTN_ERR_NULLPTR;
  if (Sk > 0 && (k == nullptr || v == nullptr)) return ATTN_ERR_NULLPTR;
  if (!aligned(q, 16) || !aligned(o, 16) || !aligned(lse, 4)) return ATTN_ERR_ALIGN;
  if (Sk > 0 && (!aligned(k, 16) || !aligned(v, 16))) return ATTN_ERR_ALIGN;
  if (kv_lens != nullptr && !aligned(kv_lens, 4)) return ATTN_ERR_ALIGN;
  // TMA strides must stay below 2^40 bytes; work units must fit an int.
  const uint64_t max_s = static_cast<uint64_t>(Sq > Sk ? Sq : Sk);
  if (static_cast<uint64_t>(H) * max_s * D * 2 >= (1ull << 40)) return ATTN_ERR_SHAPE;
  const uint64_t n_qpairs = (static_cast<uint64_t>(Sq) + kUnitRows - 1) / kUnitRows;
  if (static_cast<uint64_t>(B) * H * n_qpairs > 0x7fffffffull) return ATTN_ERR_SHAPE;

  DeviceInfo* dev = nullptr;
  attn_status st = device_info(&dev);
  if (st != ATTN_OK) return st;

  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, B, H, Sq, D)) return ATTN_ERR_CUDA;
  if (Sk > 0) {
    if (!make_map(&mk, k, B, H, Sk, D) || !make_map(&mv, v, B, H, Sk, D)) return ATTN_ERR_CUDA;
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
  p.n_qpairs = static_cast<int>(n_qpairs);
  p.total_units = static_cast<int>(static_cast<uint64_t>(B) * H * n_qpairs);
  p.c = static_cast<float>(std::fabs(static_cast<double>(scale)) * 1.4426950408889634);
  p.idesc_qk = idesc_bf16_f32(kBQ, kBK, scale < 0.0f, false);
  p.idesc_pv = idesc_bf16_f32(kBQ, D, false, true);
  p.wait_limit_ns = kWaitLimitNs;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (D == 64) {
    return causal ? launch<64, true>(*dev, 0, mq, mk, mv, p, s) : launch<64, false>(*dev, 1, mq, mk, mv, p, s);
  }
  return causal ? launch<128, true>(*dev, 2, mq, mk, mv, p, s) : launch<128, false>(*dev, 3, mq, mk, mv, p, s);
}

const char* attn_get_error_string(attn_status status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_NULLPTR: return "a required pointer is NULL";
    case ATTN_ERR_ALIGN: return "q/k/v/o must be 16-byte aligned, lse and kv_lens 4-byte aligned";
    case ATTN_ERR_SHAPE: return "invalid or too large B/H/Sq/Sk";
    case ATTN_ERR_UNSUPPORTED_D: return "head dimension D must be 64 or 128";
    case ATTN_ERR_SCALE: return "scale must be finite";
    case ATTN_ERR_CUDA: return "a CUDA call failed";
    case ATTN_ERR_DEVICE_TIMEOUT: return "a device-side wait gave up (kernel aborted its work)";
    case ATTN_ERR_UNSUPPORTED_DEVICE: return "the current device is not an sm_103 (GB300) GPU";
  }
  return "unknown status";
}

attn_status attn_check_device_status(attn_stream_t stream, uint32_t* site) {
  if (site != nullptr) *site = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
  uint32_t host[3] = {0, 0, 0};
  if (cudaMemcpyFromSymbol(host, g_attn_status, sizeof(host)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (host[0] == 0) return ATTN_OK;
  const uint32_t zero[3] = {0, 0, 0};
  if (cudaMemcpyToSymbol(g_attn_status, zero, sizeof(zero)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (site != nullptr) *site = host[1];
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

int attn_abi_version(void) { return ATTN_ABI_VERSION; }

}  // extern "C"
