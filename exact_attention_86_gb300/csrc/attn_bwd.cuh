// attn_bwd.cuh — backward pass of the exact attention on GB300 (sm_103a).
//
// Included by attn_fwd.cu inside its anonymous namespace: the backward shares
// the forward's status word, bounded waits, unit decoding and tensor maps.
//
// With P_ij = exp(s_ij - LSE_i) (s = scale * Q K^T, masked entries 0), the
// gradients of O = P V for an upstream dO are
//   dV = P^T dO,   dP = dO V^T,   dS = P * (dP - Delta),   Delta_i = <dO_i, O_i>,
//   dQ = scale * dS K,   dK = scale * dS^T Q
// (the chain rule on the softmax; the pages give the forward only).  Three
// kernels:
//   bwd_delta_kernel  Delta_i in fp32, one warp per row;
//   bwd_dq_kernel     one unit = 128 query rows of one (b, h): S and dP on
//                     the tensor cores for 64 keys at a time (two steps in
//                     flight), P and dS in the elementwise warps, dQ
//                     accumulated in TMEM over the key steps;
//   bwd_dkdv_kernel   one unit = 128 keys of one (b, h): S^T = K Q^T and
//                     dP^T = V dO^T for 64 queries at a time (two steps in
//                     flight), P^T and dS^T, then dV and dK accumulated in
//                     TMEM over the query steps.
// Both main kernels use only the operand forms of the forward: A and B
// K-major from shared memory (S, dP, S^T, dP^T) and A from TMEM with B
// MN-major from shared memory (dQ, dV, dK, like the forward's P V).

constexpr float kLog2e = 1.4426950408889634f;

enum BwdSite : uint32_t {
  kSiteBwdQFull = 33,
  kSiteBwdQEmpty = 34,
  kSiteBwdKvFull = 35,
  kSiteBwdKvEmpty = 36,
  kSiteBwdSFull = 37,
  kSiteBwdSFree = 38,
  kSiteBwdDsFull = 39,
  kSiteBwdDsFree = 40,
  kSiteBwdOutFull = 41,
};

struct BwdParams {
  Params f;              // shapes, kv_lens, n_qtiles, total_units (query or key tiles)
  const float* lse;      // [B,H,Sq] from the forward (natural log)
  const float* delta;    // [B,H,Sq] <dO_i, O_i>
  uint16_t* dq;          // [B,H,Sq,D]
  uint16_t* dk;          // [B,H,Sk,D]
  uint16_t* dv;          // [B,H,Sk,D]
  float c2;              // scale * log2(e) (signed)
  float scale;
  int n_ktiles;
};

// ---------------------------------------------------------------- Delta
template <int D>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const uint16_t* __restrict__ o,
                                                        const uint16_t* __restrict__ dout, float* __restrict__ delta,
                                                        long long rows) {
  constexpr int C = D / 32;  // elements per lane (2 or 4)
  const int lane = threadIdx.x & 31;
  const long long warp_id = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long n_warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long r = warp_id; r < rows; r += n_warps) {
    const uint16_t* po = o + r * D + lane * C;
    const uint16_t* pd = dout + r * D + lane * C;
    float acc = 0.0f;
    if constexpr (C == 4) {
      const uint2 a = __ldg(reinterpret_cast<const uint2*>(po));
      const uint2 b = __ldg(reinterpret_cast<const uint2*>(pd));
      const uint32_t av[2] = {a.x, a.y}, bv[2] = {b.x, b.y};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        acc = fmaf(__uint_as_float(av[e] << 16), __uint_as_float(bv[e] << 16), acc);
        acc = fmaf(__uint_as_float(av[e] & 0xffff0000u), __uint_as_float(bv[e] & 0xffff0000u), acc);
      }
    } else {
      const uint32_t a = __ldg(reinterpret_cast<const uint32_t*>(po));
      const uint32_t b = __ldg(reinterpret_cast<const uint32_t*>(pd));
      acc = fmaf(__uint_as_float(a << 16), __uint_as_float(b << 16), acc);
      acc = fmaf(__uint_as_float(a & 0xffff0000u), __uint_as_float(b & 0xffff0000u), acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) delta[r] = acc;
  }
}

// ------------------------------------------------------------------ dQ
// A unit is 128 query rows of one (b, h); the keys stream past in steps of 64,
// so that the S and dP of three steps fit in Tensor Memory beside the dQ
// accumulator and the tensor cores compute the next steps' products while the
// elementwise warps form dS.
constexpr int kBKDq = 64;  // keys per step

template <int D>
struct GeoDq {
  static constexpr int kTileQ = 128 * D * 2;    // Q or dO: 128 queries
  static constexpr int kTileK = kBKDq * D * 2;  // K_j or V_j: 64 keys
  static constexpr int kChunkQ = 128 * 128;     // one 128-B swizzle column of a Q/dO tile
  static constexpr int kChunkK = kBKDq * 128;   // one 128-B swizzle column of a K/V tile
  static constexpr int kChunks = D / 64;
  static constexpr int kSlots = (D == 128) ? 4 : 8;  // ring of (K_j, V_j) pairs
  static constexpr int kOffQ = 1024;
  static constexpr int kOffDo = kOffQ + kTileQ;
  static constexpr int kOffRing = kOffDo + kTileQ;
  static constexpr int kSmemBytes = kOffRing + kSlots * 2 * kTileK + 1024;
  // TMEM: step buffer b = step % kBufs holds S at [128 b, 128 b + 64) and dP
  // at [128 b + 64, 128 b + 128); each half of the elementwise warps writes dS
  // (bf16 pairs) over the first 16 of the 32 S columns it has read.  dQ at
  // 128 kBufs.
  static constexpr int kBufs = 3;
  static constexpr uint32_t kTmemDq = 128 * kBufs;
  static __device__ __forceinline__ uint32_t st_col(uint32_t b) { return 128u * b; }
  // column of the dS operand of the kk-th dQ instruction (16 keys = 8
  // columns), relative to st_col: 2 instructions per half
  static __device__ __forceinline__ uint32_t a_col(int kk) {
    return 32u * static_cast<uint32_t>(kk >> 1) + 8u * static_cast<uint32_t>(kk & 1);
  }
};
static_assert(GeoDq<128>::kSmemBytes <= 232448 && GeoDq<64>::kSmemBytes <= 232448, "shared memory");

struct CtrlDq {
  uint64_t q_full, q_empty;
  uint64_t kv_full[8], kv_empty[8];
  uint64_t st_full[3];   // S and dP of the step complete (per step buffer)
  uint64_t ds_full[3];   // dS written (8 warp arrivals)
  uint64_t buf_free[3];  // the dQ product of the step completed: its TMEM buffer is free
  uint64_t dq_full;
  uint64_t drain[2];     // one per issuing warp
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(CtrlDq) <= 1024, "control block");

// The forward's unit (head, query block, valid keys), with the keys counted in
// steps of 64: n = steps that hold a key some row of the unit may see.
template <bool CAUSAL>
__device__ __forceinline__ Unit decode_dq_unit(const Params& p, int t) {
  Unit u = decode_unit<CAUSAL>(p, t);
  int lim = u.kv;
  if (CAUSAL) lim = min(lim, u.q0 + u.rows);
  u.j0 = 0;
  u.n = u.rows > 0 ? (lim + kBKDq - 1) / kBKDq : 0;
  return u;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
                  const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                  const BwdParams bp) {
  using G = GeoDq<D>;
  const Params& p = bp.f;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  CtrlDq& ctl = *reinterpret_cast<CtrlDq*>(smem_raw + (base - raw));
  volatile int* abort_flag = &ctl.abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar_q_full = smem_addr(&ctl.q_full), bar_q_empty = smem_addr(&ctl.q_empty);
  const uint32_t bar_kv_full0 = smem_addr(&ctl.kv_full[0]), bar_kv_empty0 = smem_addr(&ctl.kv_empty[0]);
  const uint32_t bar_st_full0 = smem_addr(&ctl.st_full[0]), bar_ds_full0 = smem_addr(&ctl.ds_full[0]);
  const uint32_t bar_buf_free0 = smem_addr(&ctl.buf_free[0]);
  const uint32_t bar_dq_full = smem_addr(&ctl.dq_full);

  if (threadIdx.x == 0) {
    mbar_init(bar_q_full, 1);
    mbar_init(bar_q_empty, 1);
    for (int s = 0; s < G::kSlots; ++s) {
      mbar_init(bar_kv_full0 + 8 * s, 1);
      mbar_init(bar_kv_empty0 + 8 * s, 1);
    }
    for (int b = 0; b < G::kBufs; ++b) {
      mbar_init(bar_st_full0 + 8 * b, 1);
      mbar_init(bar_ds_full0 + 8 * b, kSoftmaxWarps);
      mbar_init(bar_buf_free0 + 8 * b, 1);
    }
    mbar_init(bar_dq_full, 1);
    mbar_init(smem_addr(&ctl.drain[0]), 1);
    mbar_init(smem_addr(&ctl.drain[1]), 1);
    ctl.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpQK) {
    tmem_alloc(smem_addr(&ctl.tmem_base), 512);
    tmem_relinquish_alloc_permit();
  }
  if (warp == kWarpLoad && lane == 0) {
    prefetch_tensor_map(&map_q);
    prefetch_tensor_map(&map_do);
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
      // -------------------------------------------------------------- TMA
      if (lane == 0) {
        const uint64_t pol_keep = l2_policy_evict_last();   // K, V: re-read by every query block of the head
        const uint64_t pol_once = l2_policy_evict_first();  // Q, dO: read once
        uint32_t ring = 0, qcount = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < t_end; t += gridDim.x) {
          const int unit = unit_at<CAUSAL>(p, t);
          if (unit >= p.total_units) continue;
          const Unit u = decode_dq_unit<CAUSAL>(p, unit);
          if (u.n == 0) continue;
          if (!wait_phase(bar_q_empty, (qcount & 1u) ^ 1u, abort_flag, kSiteBwdQEmpty, limit)) { ok = false; break; }
          mbar_arrive_expect_tx(bar_q_full, 2 * G::kTileQ);
          for (int c = 0; c < G::kChunks; ++c) {
            tma_load_4d_hint(base + G::kOffQ + c * G::kChunkQ, &map_q, bar_q_full, c * 64, u.q0, u.h, u.b,
                             pol_once);
            tma_load_4d_hint(base + G::kOffDo + c * G::kChunkQ, &map_do, bar_q_full, c * 64, u.q0, u.h, u.b,
                             pol_once);
          }
          ++qcount;
          for (int j = 0; ok && j < u.n; ++j) {
            const uint32_t slot = ring % G::kSlots;
            const uint32_t ph = (ring / G::kSlots) & 1u;
            if (!wait_phase(bar_kv_empty0 + 8 * slot, ph ^ 1u, abort_flag, kSiteBwdKvEmpty, limit)) {
              ok = false;
              break;
            }
            const uint32_t full = bar_kv_full0 + 8 * slot;
            mbar_arrive_expect_tx(full, 2 * G::kTileK);
            const uint32_t dst = base + G::kOffRing + slot * 2 * G::kTileK;
            const int key0 = (u.j0 + j) * kBKDq;
            for (int c = 0; c < G::kChunks; ++c) {
              tma_load_4d_hint(dst + c * G::kChunkK, &map_k, full, c * 64, key0, u.h, u.b, pol_keep);
              tma_load_4d_hint(dst + G::kTileK + c * G::kChunkK, &map_v, full, c * 64, key0, u.h, u.b, pol_keep);
            }
            ++ring;
          }
        }
        if (!ok) {
          if (qcount > 0) wait_phase_drain(bar_q_full, (qcount - 1) & 1u);
          for (uint32_t s = 0; s < (uint32_t)G::kSlots && s < ring; ++s) {
            const uint32_t last = ring - 1 - ((ring - 1 - s) % G::kSlots);
            wait_phase_drain(bar_kv_full0 + 8 * s, (last / G::kSlots) & 1u);
          }
        }
        // the issuers' last commit arrivals land asynchronously: wait for them
        if (qcount > 0) wait_phase_drain(bar_q_empty, (qcount - 1) & 1u);
        for (uint32_t s = 0; s < (uint32_t)G::kSlots && s < ring; ++s) {
          const uint32_t last = ring - 1 - ((ring - 1 - s) % G::kSlots);
          wait_phase_drain(bar_kv_empty0 + 8 * s, (last / G::kSlots) & 1u);
        }
      }
      __syncwarp();
    } else if (warp == kWarpQK) {
      // ---------------------------------------------------- S, dP issuer
      // Per step t: S = Q K_t^T and dP = dO V_t^T into step buffer t % kBufs,
      // once the dQ product of step t - kBufs has released it.
      const uint32_t idesc_s = idesc_bf16_f32(kBQ, kBKDq, false, false);
      const uint32_t qa = base + G::kOffQ, da = base + G::kOffDo;
      uint32_t tcount = 0, qcount = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < t_end; t += gridDim.x) {
        const int unit = unit_at<CAUSAL>(p, t);
        if (unit >= p.total_units) continue;
        const Unit u = decode_dq_unit<CAUSAL>(p, unit);
        if (u.n == 0) continue;
        if (!wait_warp(bar_q_full, qcount & 1u, abort_flag, kSiteBwdQFull, limit)) { ok = false; break; }
        ++qcount;
        for (int j = 0; j < u.n; ++j) {
          const uint32_t tt = tcount + j;
          const uint32_t b = tt % G::kBufs;
          const uint32_t slot = tt % G::kSlots;
          if (!wait_warp(bar_kv_full0 + 8 * slot, (tt / G::kSlots) & 1u, abort_flag, kSiteBwdKvFull, limit)) {
            ok = false;
            break;
          }
          if (tt >= static_cast<uint32_t>(G::kBufs) &&
              !wait_warp(bar_buf_free0 + 8 * b, (tt / G::kBufs - 1) & 1u, abort_flag, kSiteBwdSFree, limit)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t ka = base + G::kOffRing + slot * 2 * G::kTileK;
          const uint32_t va = ka + G::kTileK;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off_q = (kk >> 2) * G::kChunkQ + (kk & 3) * 32;
            const uint32_t off_k = (kk >> 2) * G::kChunkK + (kk & 3) * 32;
            mma_ss_elect(tmem + G::st_col(b), sdesc_sw128(qa + off_q, 16, 1024), sdesc_sw128(ka + off_k, 16, 1024),
                         idesc_s, kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off_q = (kk >> 2) * G::kChunkQ + (kk & 3) * 32;
            const uint32_t off_k = (kk >> 2) * G::kChunkK + (kk & 3) * 32;
            mma_ss_elect(tmem + G::st_col(b) + 64, sdesc_sw128(da + off_q, 16, 1024),
                         sdesc_sw128(va + off_k, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
          }
          mma_commit_elect(bar_st_full0 + 8 * b);
          if (j == u.n - 1) mma_commit_elect(bar_q_empty);  // Q and dO are done after the unit's last S, dP
        }
        if (!ok) break;
        tcount += u.n;
      }
      const uint32_t bar_d = smem_addr(&ctl.drain[0]);
      mma_commit_elect(bar_d);
      wait_phase_drain(bar_d, 0);
    } else if (warp == kWarpPV) {
      // --------------------------------------------------------- dQ issuer
      // Per step t, once the elementwise warps have written dS_t: dQ +=
      // dS_t K_t; its commit frees the step's TMEM buffer and ring slot (V_t
      // was read by dP_t, which completed before the elementwise warps began).
      const uint32_t idesc_q = idesc_bf16_f32(kBQ, D, false, true);
      uint32_t tcount = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < t_end; t += gridDim.x) {
        const int unit = unit_at<CAUSAL>(p, t);
        if (unit >= p.total_units) continue;
        const Unit u = decode_dq_unit<CAUSAL>(p, unit);
        if (u.n == 0) continue;
        for (int j = 0; j < u.n; ++j) {
          const uint32_t tt = tcount + j;
          const uint32_t b = tt % G::kBufs;
          const uint32_t slot = tt % G::kSlots;
          if (!wait_warp(bar_ds_full0 + 8 * b, (tt / G::kBufs) & 1u, abort_flag, kSiteBwdDsFull, limit)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t ka = base + G::kOffRing + slot * 2 * G::kTileK;
#pragma unroll
          for (int kk = 0; kk < kBKDq / 16; ++kk)
            mma_ts_elect(tmem + G::kTmemDq, tmem + G::st_col(b) + G::a_col(kk),
                         sdesc_sw128(ka + kk * 16 * 128, G::kChunkK, 1024), idesc_q, (j == 0 && kk == 0) ? 0u : 1u);
          mma_commit_elect(bar_buf_free0 + 8 * b);
          mma_commit_elect(bar_kv_empty0 + 8 * slot);
        }
        if (!ok) break;
        mma_commit_elect(bar_dq_full);
        tcount += u.n;
      }
      const uint32_t bar_d = smem_addr(&ctl.drain[1]);
      mma_commit_elect(bar_d);
      wait_phase_drain(bar_d, 0);
      if (ok) {
        for (uint32_t back = 1; back <= static_cast<uint32_t>(G::kBufs) && back <= tcount; ++back) {
          const uint32_t t = tcount - back;
          wait_phase_drain(bar_buf_free0 + 8 * (t % G::kBufs), (t / G::kBufs) & 1u);
        }
      }
    }
  } else {
    regs_increase<kRegsSoftmax>();
    // ------------------------------------------------------- elementwise
    // Two threads per query row: warps 0-3 own key columns 0-31 of each step
    // and dQ columns [0, D/2), warps 4-7 the rest.  Each warp reads and
    // writes only its own TMEM columns, so the warps never wait for one
    // another and a failed wait lets a warp leave on its own.
    const int half = warp >> 2;
    const int r = threadIdx.x & (kBQ - 1);
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t tcount = 0, ucount = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < t_end; t += gridDim.x) {
      const int unit = unit_at<CAUSAL>(p, t);
      if (unit >= p.total_units) continue;
      const Unit u = decode_dq_unit<CAUSAL>(p, unit);
      const int row = u.q0 + r;
      const bool row_ok = row < p.Sq;
      const size_t row_index = (static_cast<size_t>(u.b) * p.H + u.h) * static_cast<size_t>(p.Sq) + row;
      uint16_t* dq_dst = bp.dq + row_index * D + (D / 2) * half;
      if (u.n == 0) {  // no valid key for any row: dQ = 0
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(dq_dst);
#pragma unroll
          for (int q = 0; q < D / 16; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      const float lse_i = row_ok ? __ldg(bp.lse + row_index) : -INFINITY;
      const bool live = row_ok && lse_i != -INFINITY;
      const float lse2 = live ? lse_i * kLog2e : 0.0f;
      const float delta_i = row_ok ? __ldg(bp.delta + row_index) : 0.0f;
      const bool rows_tail = u.q0 + kBQ > p.Sq;
      for (int j = 0; j < u.n; ++j) {
        const uint32_t tt = tcount + j;
        const uint32_t b = tt % G::kBufs;
        const int k0 = (u.j0 + j) * kBKDq;
        // key column c of this half is k0 + 32*half + c: valid below kv and,
        // causal, up to the row
        const bool masked = !live || rows_tail || (k0 + kBKDq > u.kv) || (CAUSAL && k0 + kBKDq - 1 > u.q0);
        int climit = u.kv - k0;
        if (CAUSAL) climit = min(climit, row - k0 + 1);
        climit = live ? climit - 32 * half : 0;
        if (!wait_warp(bar_st_full0 + 8 * b, (tt / G::kBufs) & 1u, abort_flag, kSiteBwdSFull, limit)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t tS = tmem + lane_off + G::st_col(b) + 32u * half;
        uint32_t s[32], dp[32];
        tmem_ld_32x32b_x32(tS, s);
        tmem_ld_32x32b_x32(tS + 64, dp);
        tmem_ld_wait_x32(s);
        tmem_ld_wait_x32(dp);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float s0 = __uint_as_float(s[2 * e]), s1 = __uint_as_float(s[2 * e + 1]);
          const float d0 = __uint_as_float(dp[2 * e]), d1 = __uint_as_float(dp[2 * e + 1]);
          float p0 = ex2_approx(fmaf(s0, bp.c2, -lse2));
          float p1 = ex2_approx(fmaf(s1, bp.c2, -lse2));
          if (masked) {
            p0 = (2 * e < climit) ? p0 : 0.0f;
            p1 = (2 * e + 1 < climit) ? p1 : 0.0f;
          }
          pk[e] = pack_bf16x2(p0 * (d0 - delta_i), p1 * (d1 - delta_i));
        }
        tmem_st_32x32b_x16(tS, pk);  // dS over the S columns just read
        tmem_st_wait();
        warp_arrive_after_tc(bar_ds_full0 + 8 * b, lane);
      }
      if (!ok) break;
      tcount += u.n;
      if (!wait_warp(bar_dq_full, ucount & 1u, abort_flag, kSiteBwdOutFull, limit)) { ok = false; break; }
      ++ucount;
      tc_fence_after_sync();
      const uint32_t tQ = tmem + lane_off + G::kTmemDq + (D / 2) * half;
#pragma unroll
      for (int q = 0; q < D / 64; ++q) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tQ + q * 32, o);
        tmem_ld_wait_x32(o);
        if (row_ok) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * bp.scale, __uint_as_float(o[2 * e + 1]) * bp.scale);
          uint4* dst = reinterpret_cast<uint4*>(dq_dst + q * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
      }
      // the next unit's first dQ product overwrites the accumulator only after
      // every elementwise warp has arrived on ds_full for it, which comes after this
      tc_fence_before_sync();
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpQK) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// --------------------------------------------------------------- dK, dV
// A unit is 128 keys of one (b, h); the query rows stream past it in steps of
// 64, so that the two products of a step (S^T, dP^T: 64 columns each) fit
// twice in Tensor Memory beside the dV and dK accumulators, and the tensor
// cores compute the next step's products while the elementwise warps turn the
// current ones into P^T and dS^T.
constexpr int kBQKv = 64;  // query rows per step

template <int D>
struct GeoKv {
  static constexpr int kTileK = 128 * D * 2;     // K or V: 128 keys
  static constexpr int kTileQ = kBQKv * D * 2;   // Q_i or dO_i: 64 queries
  static constexpr int kChunkK = 128 * 128;      // one 128-B swizzle column of a K/V tile
  static constexpr int kChunkQ = kBQKv * 128;    // one 128-B swizzle column of a Q/dO tile
  static constexpr int kChunks = D / 64;
  static constexpr int kSlots = (D == 128) ? 4 : 8;  // ring of (Q_i, dO_i) pairs
  static constexpr int kOffStat = 1024;  // per warp and step parity: LSE*log2e[32], Delta[32] (4 KB)
  static constexpr int kOffK = 5120;
  static constexpr int kOffV = kOffK + kTileK;
  static constexpr int kOffRing = kOffV + kTileK;
  static constexpr int kSmemBytes = kOffRing + kSlots * 2 * kTileQ + 1024;
  // TMEM: step parity b holds S^T at [128 b, 128 b + 64) and dP^T at
  // [128 b + 64, 128 b + 128).  Each half of the elementwise warps reads its 32
  // columns of both and writes P^T and dS^T (bf16 pairs) over the first 16 of
  // them, so no half writes where the other reads.  dV at 256, dK at 256 + D.
  static constexpr uint32_t kTmemDv = 256, kTmemDk = 256 + D;
  static __device__ __forceinline__ uint32_t st_col(uint32_t b) { return 128u * b; }
  // column of the A operand (P^T or dS^T) of the kk-th product instruction
  // (16 queries = 8 columns), relative to st_col: 2 instructions per half
  static __device__ __forceinline__ uint32_t a_col(int kk) {
    return 32u * static_cast<uint32_t>(kk >> 1) + 8u * static_cast<uint32_t>(kk & 1);
  }
};
static_assert(GeoKv<128>::kSmemBytes <= 232448 && GeoKv<64>::kSmemBytes <= 232448, "shared memory");
static_assert(8 * 2 * 64 * 4 <= GeoKv<128>::kOffK - GeoKv<128>::kOffStat, "staging area");

struct CtrlKv {
  uint64_t kv_full, kv_empty;
  uint64_t qd_full[8], qd_empty[8];
  uint64_t st_full[2];  // S^T and dP^T of the step complete
  uint64_t pd_full[2];  // P^T and dS^T written (8 warp arrivals)
  uint64_t s_free[2];   // the dV product of the step completed (its S^T columns are free)
  uint64_t d_free[2];   // the dK product completed (dP^T columns and the ring slot are free)
  uint64_t out_full;
  uint64_t drain[2];  // one per issuing warp
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(CtrlKv) <= 1024, "control block");

struct KvUnit {
  int b, h, key0, rows_k;  // rows_k: keys of the tile that exist (< Sk)
  int kv;                  // valid keys of the batch entry
  int i0, n;               // first query step and number of steps (0: no gradient)
};

template <bool CAUSAL>
__device__ __forceinline__ KvUnit decode_kv_unit(const BwdParams& bp, int t) {
  const Params& p = bp.f;
  KvUnit u;
  const int bh_count = p.B * p.H;
  int kt, bh;
  if (CAUSAL) {  // longest first: key tiles from the start of the sequence
    kt = t / bh_count;
    bh = t % bh_count;
  } else {       // consecutive units share a head, so its Q and dO stay hot in L2
    kt = t % bp.n_ktiles;
    bh = t / bp.n_ktiles;
  }
  u.b = bh / p.H;
  u.h = bh % p.H;
  u.key0 = kt * kBK;
  u.rows_k = max(min(kBK, p.Sk - u.key0), 0);
  int kv = p.Sk;
  if (p.kv_lens != nullptr) kv = min(max(__ldg(p.kv_lens + u.b), 0), p.Sk);
  u.kv = kv;
  u.i0 = CAUSAL ? u.key0 / kBQKv : 0;  // query rows below key0 see none of these keys
  u.n = (u.key0 < kv && u.rows_k > 0) ? max(p.n_qtiles - u.i0, 0) : 0;  // n_qtiles counts 64-row steps here
  return u;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
                    const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                    const BwdParams bp) {
  using G = GeoKv<D>;
  const Params& p = bp.f;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  CtrlKv& ctl = *reinterpret_cast<CtrlKv*>(base_ptr);
  volatile int* abort_flag = &ctl.abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar_kv_full = smem_addr(&ctl.kv_full), bar_kv_empty = smem_addr(&ctl.kv_empty);
  const uint32_t bar_qd_full0 = smem_addr(&ctl.qd_full[0]), bar_qd_empty0 = smem_addr(&ctl.qd_empty[0]);
  const uint32_t bar_st_full0 = smem_addr(&ctl.st_full[0]), bar_pd_full0 = smem_addr(&ctl.pd_full[0]);
  const uint32_t bar_s_free0 = smem_addr(&ctl.s_free[0]), bar_d_free0 = smem_addr(&ctl.d_free[0]);
  const uint32_t bar_out_full = smem_addr(&ctl.out_full);

  if (threadIdx.x == 0) {
    mbar_init(bar_kv_full, 1);
    mbar_init(bar_kv_empty, 1);
    for (int s = 0; s < G::kSlots; ++s) {
      mbar_init(bar_qd_full0 + 8 * s, 1);
      mbar_init(bar_qd_empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_st_full0 + 8 * b, 1);
      mbar_init(bar_pd_full0 + 8 * b, kSoftmaxWarps);
      mbar_init(bar_s_free0 + 8 * b, 1);
      mbar_init(bar_d_free0 + 8 * b, 1);
    }
    mbar_init(bar_out_full, 1);
    mbar_init(smem_addr(&ctl.drain[0]), 1);
    mbar_init(smem_addr(&ctl.drain[1]), 1);
    ctl.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpQK) {
    tmem_alloc(smem_addr(&ctl.tmem_base), 512);
    tmem_relinquish_alloc_permit();
  }
  if (warp == kWarpLoad && lane == 0) {
    prefetch_tensor_map(&map_q);
    prefetch_tensor_map(&map_do);
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
      // -------------------------------------------------------------- TMA
      if (lane == 0) {
        const uint64_t pol_keep = l2_policy_evict_last();   // Q, dO: re-read by every key tile of the head
        const uint64_t pol_once = l2_policy_evict_first();  // K, V: read once
        uint32_t ring = 0, ucount = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < t_end; t += gridDim.x) {
          const int unit = unit_at<CAUSAL>(p, t);
          if (unit >= p.total_units) continue;
          const KvUnit u = decode_kv_unit<CAUSAL>(bp, unit);
          if (u.n == 0) continue;
          if (!wait_phase(bar_kv_empty, (ucount & 1u) ^ 1u, abort_flag, kSiteBwdKvEmpty, limit)) { ok = false; break; }
          mbar_arrive_expect_tx(bar_kv_full, 2 * G::kTileK);
          for (int c = 0; c < G::kChunks; ++c) {
            tma_load_4d_hint(base + G::kOffK + c * G::kChunkK, &map_k, bar_kv_full, c * 64, u.key0, u.h, u.b,
                             pol_once);
            tma_load_4d_hint(base + G::kOffV + c * G::kChunkK, &map_v, bar_kv_full, c * 64, u.key0, u.h, u.b,
                             pol_once);
          }
          ++ucount;
          for (int i = 0; ok && i < u.n; ++i) {
            const uint32_t slot = ring % G::kSlots;
            const uint32_t ph = (ring / G::kSlots) & 1u;
            if (!wait_phase(bar_qd_empty0 + 8 * slot, ph ^ 1u, abort_flag, kSiteBwdQEmpty, limit)) {
              ok = false;
              break;
            }
            const uint32_t full = bar_qd_full0 + 8 * slot;
            mbar_arrive_expect_tx(full, 2 * G::kTileQ);
            const uint32_t dst = base + G::kOffRing + slot * 2 * G::kTileQ;
            const int q0 = (u.i0 + i) * kBQKv;
            for (int c = 0; c < G::kChunks; ++c) {
              tma_load_4d_hint(dst + c * G::kChunkQ, &map_q, full, c * 64, q0, u.h, u.b, pol_keep);
              tma_load_4d_hint(dst + G::kTileQ + c * G::kChunkQ, &map_do, full, c * 64, q0, u.h, u.b, pol_keep);
            }
            ++ring;
          }
        }
        if (!ok) {
          if (ucount > 0) wait_phase_drain(bar_kv_full, (ucount - 1) & 1u);
          for (uint32_t s = 0; s < (uint32_t)G::kSlots && s < ring; ++s) {
            const uint32_t last = ring - 1 - ((ring - 1 - s) % G::kSlots);
            wait_phase_drain(bar_qd_full0 + 8 * s, (last / G::kSlots) & 1u);
          }
        }
        if (ucount > 0) wait_phase_drain(bar_kv_empty, (ucount - 1) & 1u);
        for (uint32_t s = 0; s < (uint32_t)G::kSlots && s < ring; ++s) {
          const uint32_t last = ring - 1 - ((ring - 1 - s) % G::kSlots);
          wait_phase_drain(bar_qd_empty0 + 8 * s, (last / G::kSlots) & 1u);
        }
      }
      __syncwarp();
    } else if (warp == kWarpQK) {
      // ------------------------------------------------- S^T, dP^T issuer
      // Per step t: S^T_t once the dV product of step t-2 has released its
      // columns, dP^T_t once the dK product of t-2 has, one commit for both.
      // The products have their own issuing warp, so this one runs ahead
      // while they wait for the elementwise warps.
      const uint32_t idesc_s = idesc_bf16_f32(kBK, kBQKv, false, false);
      const uint32_t ka = base + G::kOffK, va = base + G::kOffV;
      uint32_t tcount = 0, ucount = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < t_end; t += gridDim.x) {
        const int unit = unit_at<CAUSAL>(p, t);
        if (unit >= p.total_units) continue;
        const KvUnit u = decode_kv_unit<CAUSAL>(bp, unit);
        if (u.n == 0) continue;
        if (!wait_warp(bar_kv_full, ucount & 1u, abort_flag, kSiteBwdKvFull, limit)) { ok = false; break; }
        ++ucount;
        for (int i = 0; i < u.n; ++i) {
          const uint32_t tt = tcount + i;
          const uint32_t b = tt & 1u;
          const uint32_t slot = tt % G::kSlots;
          if (!wait_warp(bar_qd_full0 + 8 * slot, (tt / G::kSlots) & 1u, abort_flag, kSiteBwdQFull, limit)) {
            ok = false;
            break;
          }
          const uint32_t prev_use = ((tt >> 1) - 1) & 1u;  // parity of step tt-2's release
          if (tt >= 2 && !wait_warp(bar_s_free0 + 8 * b, prev_use, abort_flag, kSiteBwdSFree, limit)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t qa = base + G::kOffRing + slot * 2 * G::kTileQ;
          const uint32_t da = qa + G::kTileQ;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off_k = (kk >> 2) * G::kChunkK + (kk & 3) * 32;
            const uint32_t off_q = (kk >> 2) * G::kChunkQ + (kk & 3) * 32;
            mma_ss_elect(tmem + G::st_col(b), sdesc_sw128(ka + off_k, 16, 1024), sdesc_sw128(qa + off_q, 16, 1024),
                         idesc_s, kk > 0 ? 1u : 0u);
          }
          if (tt >= 2 && !wait_warp(bar_d_free0 + 8 * b, prev_use, abort_flag, kSiteBwdDsFree, limit)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off_k = (kk >> 2) * G::kChunkK + (kk & 3) * 32;
            const uint32_t off_q = (kk >> 2) * G::kChunkQ + (kk & 3) * 32;
            mma_ss_elect(tmem + G::st_col(b) + 64, sdesc_sw128(va + off_k, 16, 1024),
                         sdesc_sw128(da + off_q, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
          }
          mma_commit_elect(bar_st_full0 + 8 * b);
        }
        if (!ok) break;
        tcount += u.n;
      }
      // every MMA of this warp has completed before TMEM is released
      const uint32_t bar_d = smem_addr(&ctl.drain[0]);
      mma_commit_elect(bar_d);
      wait_phase_drain(bar_d, 0);
    } else if (warp == kWarpPV) {
      // ------------------------------------------------ dV, dK issuer
      // Per step t, once the elementwise warps have written P^T and dS^T:
      // dV += P^T dO_t (its commit releases the S^T columns), dK += dS^T Q_t
      // (releases the dP^T columns and the ring slot).  After a unit's last
      // step: the accumulators are complete, and K/V may be replaced (the
      // S^T and dP^T products that read them completed before the elementwise
      // warps could finish that step).
      const uint32_t idesc_o = idesc_bf16_f32(kBK, D, false, true);
      uint32_t tcount = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < t_end; t += gridDim.x) {
        const int unit = unit_at<CAUSAL>(p, t);
        if (unit >= p.total_units) continue;
        const KvUnit u = decode_kv_unit<CAUSAL>(bp, unit);
        if (u.n == 0) continue;
        for (int i = 0; i < u.n; ++i) {
          const uint32_t tt = tcount + i;
          const uint32_t b = tt & 1u;
          const uint32_t slot = tt % G::kSlots;
          if (!wait_warp(bar_pd_full0 + 8 * b, (tt >> 1) & 1u, abort_flag, kSiteBwdDsFull, limit)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t qa = base + G::kOffRing + slot * 2 * G::kTileQ;
          const uint32_t da = qa + G::kTileQ;
#pragma unroll
          for (int kk = 0; kk < kBQKv / 16; ++kk)
            mma_ts_elect(tmem + G::kTmemDv, tmem + G::st_col(b) + G::a_col(kk),
                         sdesc_sw128(da + kk * 16 * 128, G::kChunkQ, 1024), idesc_o, (i == 0 && kk == 0) ? 0u : 1u);
          mma_commit_elect(bar_s_free0 + 8 * b);
#pragma unroll
          for (int kk = 0; kk < kBQKv / 16; ++kk)
            mma_ts_elect(tmem + G::kTmemDk, tmem + G::st_col(b) + 64 + G::a_col(kk),
                         sdesc_sw128(qa + kk * 16 * 128, G::kChunkQ, 1024), idesc_o, (i == 0 && kk == 0) ? 0u : 1u);
          mma_commit_elect(bar_d_free0 + 8 * b);
          mma_commit_elect(bar_qd_empty0 + 8 * slot);
        }
        if (!ok) break;
        mma_commit_elect(bar_out_full);
        mma_commit_elect(bar_kv_empty);
        tcount += u.n;
      }
      // every product has completed (and its commits have landed) before
      // TMEM is released and the CTA exits
      const uint32_t bar_d = smem_addr(&ctl.drain[1]);
      mma_commit_elect(bar_d);
      wait_phase_drain(bar_d, 0);
      if (ok) {
        for (uint32_t back = 1; back <= 2 && back <= tcount; ++back) {
          const uint32_t t = tcount - back;
          wait_phase_drain(bar_s_free0 + 8 * (t & 1u), (t >> 1) & 1u);
          wait_phase_drain(bar_d_free0 + 8 * (t & 1u), (t >> 1) & 1u);
        }
      }
    }
  } else {
    regs_increase<kRegsSoftmax>();
    // ------------------------------------------------------- elementwise
    // Two threads per key row: warps 0-3 own query columns 0-31 of each step
    // and dK/dV columns [0, D/2), warps 4-7 the rest.  The warps never wait
    // for one another: each reads and writes only its own TMEM columns and
    // stages its own LSE and Delta values, so a failed wait lets a warp leave
    // on its own.
    const int half = warp >> 2;
    const int r = threadIdx.x & (kBK - 1);
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    float* stage = reinterpret_cast<float*>(base_ptr + G::kOffStat) + warp * 2 * 64;
    uint32_t tcount = 0, ucount = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < t_end; t += gridDim.x) {
      const int unit = unit_at<CAUSAL>(p, t);
      if (unit >= p.total_units) continue;
      const KvUnit u = decode_kv_unit<CAUSAL>(bp, unit);
      const int key = u.key0 + r;
      const bool key_exists = r < u.rows_k;
      const bool key_ok = key < u.kv;
      const size_t key_index = (static_cast<size_t>(u.b) * p.H + u.h) * static_cast<size_t>(p.Sk) + key;
      uint16_t* dk_dst = bp.dk + key_index * D + (D / 2) * half;
      uint16_t* dv_dst = bp.dv + key_index * D + (D / 2) * half;
      if (u.n == 0) {  // no query sees these keys (or none is valid): dK = dV = 0
        if (key_exists) {
#pragma unroll
          for (int q = 0; q < D / 16; ++q) {
            reinterpret_cast<uint4*>(dk_dst)[q] = make_uint4(0u, 0u, 0u, 0u);
            reinterpret_cast<uint4*>(dv_dst)[q] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        continue;
      }
      const size_t head_row0 = (static_cast<size_t>(u.b) * p.H + u.h) * static_cast<size_t>(p.Sq);
      // LSE (base 2) and Delta of this half's 32 queries of a step, one per
      // lane, fetched a step ahead; a query past Sq or without a valid key
      // gets LSE = +inf, so its P is 0
      float lse_raw = -INFINITY, del_raw = 0.0f;
      auto fetch = [&](int step) {
        const int q = (u.i0 + step) * kBQKv + 32 * half + lane;
        lse_raw = -INFINITY;
        del_raw = 0.0f;
        if (q < p.Sq) {
          lse_raw = __ldg(bp.lse + head_row0 + q);
          del_raw = __ldg(bp.delta + head_row0 + q);
        }
      };
      fetch(0);
      for (int i = 0; i < u.n; ++i) {
        const uint32_t tt = tcount + i;
        const uint32_t b = tt & 1u;
        const int q0 = (u.i0 + i) * kBQKv;
        // into the warp's staging slot of this step's parity, negated:
        // -LSE*log2e (-inf for no key: P = 0) and -Delta
        stage[b * 64 + lane] = (lse_raw == -INFINITY) ? -INFINITY : -lse_raw * kLog2e;
        stage[b * 64 + 32 + lane] = -del_raw;
        __syncwarp();
        if (i + 1 < u.n) fetch(i + 1);
        // query column c of this half is q0 + 32*half + c; key <= query for causal
        const bool masked = !key_ok || (CAUSAL && q0 < u.key0 + kBK - 1);
        const int cstart = key_ok ? (CAUSAL ? key - q0 - 32 * half : 0) : 32;  // first valid column
        if (!wait_warp(bar_st_full0 + 8 * b, (tt >> 1) & 1u, abort_flag, kSiteBwdSFull, limit)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t tS = tmem + lane_off + G::st_col(b) + 32u * half;
        const uint32_t tD = tS + 64u;
        uint32_t s[32], dp[32];
        tmem_ld_32x32b_x32(tS, s);
        tmem_ld_32x32b_x32(tD, dp);
        tmem_ld_wait_x32(s);
        tmem_ld_wait_x32(dp);
        // pairs of columns: -LSE*log2e and -Delta come as packed pairs
        const uint64_t* nlse2 = reinterpret_cast<const uint64_t*>(stage + b * 64);
        const uint64_t* ndel2 = nlse2 + 16;
        const uint64_t c2x2 = f2_pack(bp.c2, bp.c2);
        uint32_t pk[16], ds_pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1])), c2x2, nlse2[e]), x0,
                    x1);
          float p0 = ex2_approx(x0);
          float p1 = ex2_approx(x1);
          if (masked) {
            p0 = (2 * e >= cstart) ? p0 : 0.0f;
            p1 = (2 * e + 1 >= cstart) ? p1 : 0.0f;
          }
          pk[e] = pack_bf16x2(p0, p1);
          const uint64_t diff = f2_add(f2_pack(__uint_as_float(dp[2 * e]), __uint_as_float(dp[2 * e + 1])), ndel2[e]);
          float g0, g1;
          f2_unpack(f2_mul(f2_pack(p0, p1), diff), g0, g1);
          ds_pk[e] = pack_bf16x2(g0, g1);
        }
        tmem_st_32x32b_x16(tS, pk);
        tmem_st_32x32b_x16(tD, ds_pk);
        tmem_st_wait();
        warp_arrive_after_tc(bar_pd_full0 + 8 * b, lane);
      }
      if (!ok) break;
      tcount += u.n;
      if (!wait_warp(bar_out_full, ucount & 1u, abort_flag, kSiteBwdOutFull, limit)) { ok = false; break; }
      ++ucount;
      tc_fence_after_sync();
#pragma unroll
      for (int which = 0; which < 2; ++which) {  // dV, then dK (times scale)
        const uint32_t tA = tmem + lane_off + (which ? G::kTmemDk : G::kTmemDv) + (D / 2) * half;
        const float mul = which ? bp.scale : 1.0f;
        uint16_t* dst16 = which ? dk_dst : dv_dst;
#pragma unroll
        for (int q = 0; q < D / 64; ++q) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tA + q * 32, o);
          tmem_ld_wait_x32(o);
          if (key_exists) {
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              w[e] = key_ok ? pack_bf16x2(__uint_as_float(o[2 * e]) * mul, __uint_as_float(o[2 * e + 1]) * mul) : 0u;
            uint4* dst = reinterpret_cast<uint4*>(dst16 + q * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
          }
        }
      }
      // the next unit's first dV/dK product overwrites the accumulators only
      // after every elementwise warp has arrived on pd_full for it, which
      // comes after this
      tc_fence_before_sync();
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpQK) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ host
size_t bwd_delta_bytes(int B, int H, int Sq) {
  return round_up_256(static_cast<size_t>(B) * H * Sq * sizeof(float));
}

template <int D, bool CAUSAL>
attn_status launch_bwd(DeviceInfo& dev, int idx, const CUtensorMap& mq, const CUtensorMap& mdo,
                       const CUtensorMap& mq64, const CUtensorMap& mdo64, const CUtensorMap& mk,
                       const CUtensorMap& mv, const CUtensorMap& mk64, const CUtensorMap& mv64, const BwdParams& bq,
                       const BwdParams& bk, cudaStream_t stream) {
  auto kq = bwd_dq_kernel<D, CAUSAL>;
  auto kk = bwd_dkdv_kernel<D, CAUSAL>;
  constexpr int smem_q = GeoDq<D>::kSmemBytes;
  constexpr int smem_k = GeoKv<D>::kSmemBytes;
  if (!dev.bwd_smem_set[idx].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_q) != cudaSuccess ||
        cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_k) != cudaSuccess)
      return ATTN_ERR_CUDA;
    dev.bwd_smem_set[idx].store(true, std::memory_order_release);
  }
  if (bq.f.total_units > 0) {
    const int grid = bq.f.total_units < dev.num_sms ? bq.f.total_units : dev.num_sms;
    BwdParams bqd = bq;
    bqd.f = with_divisors(bq.f, grid);
    kq<<<grid, kThreads, smem_q, stream>>>(mq, mdo, mk64, mv64, bqd);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  }
  if (bk.f.total_units > 0) {
    const int grid = bk.f.total_units < dev.num_sms ? bk.f.total_units : dev.num_sms;
    BwdParams bkd = bk;
    bkd.f = with_divisors(bk.f, grid);
    kk<<<grid, kThreads, smem_k, stream>>>(mq64, mdo64, mk, mv, bkd);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

attn_status run_backward(DeviceInfo& dev, const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv, int B, int H, int Sq,
                         int Sk, int D, float scale, int causal, const int32_t* kv_lens, float* delta,
                         cudaStream_t s) {
  if (Sq == 0) {  // no query: dK = dV = 0
    const size_t bytes = static_cast<size_t>(B) * H * Sk * D * 2;
    if (cudaMemsetAsync(dk, 0, bytes, s) != cudaSuccess || cudaMemsetAsync(dv, 0, bytes, s) != cudaSuccess)
      return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  if (Sk == 0) {  // no key: dQ = 0
    if (cudaMemsetAsync(dq, 0, static_cast<size_t>(B) * H * Sq * D * 2, s) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  // Delta_i = <dO_i, O_i>
  const long long rows = static_cast<long long>(B) * H * Sq;
  long long blocks = (rows + 7) / 8;
  const long long max_blocks = static_cast<long long>(dev.num_sms) * 8;
  if (blocks > max_blocks) blocks = max_blocks;
  if (D == 64)
    bwd_delta_kernel<64><<<static_cast<int>(blocks), 256, 0, s>>>(static_cast<const uint16_t*>(o),
                                                                   static_cast<const uint16_t*>(dout), delta, rows);
  else
    bwd_delta_kernel<128><<<static_cast<int>(blocks), 256, 0, s>>>(static_cast<const uint16_t*>(o),
                                                                    static_cast<const uint16_t*>(dout), delta, rows);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;

  // 128-row boxes for what a kernel holds for a whole unit, 64-row boxes for
  // what streams past it in steps
  CUtensorMap mq, mdo, mq64, mdo64, mk, mv, mk64, mv64;
  if (!make_map(&mq, q, B, H, Sq, D) || !make_map(&mdo, dout, B, H, Sq, D) ||
      !make_map(&mq64, q, B, H, Sq, D, kBQKv) || !make_map(&mdo64, dout, B, H, Sq, D, kBQKv) ||
      !make_map(&mk, k, B, H, Sk, D) || !make_map(&mv, v, B, H, Sk, D) ||
      !make_map(&mk64, k, B, H, Sk, D, kBKDq) || !make_map(&mv64, v, B, H, Sk, D, kBKDq))
    return ATTN_ERR_CUDA;
  BwdParams bq;
  Params& f = bq.f;
  f.o = nullptr;
  f.lse = nullptr;
  f.kv_lens = kv_lens;
  f.B = B;
  f.H = H;
  f.Sq = Sq;
  f.Sk = Sk;
  f.n_qtiles = (Sq + kBQ - 1) / kBQ;
  f.head_group = head_group_for(B * H, Sk, D, 2);
  f.num_splits = 1;
  f.total_units = static_cast<int>(static_cast<int64_t>(B) * H * f.n_qtiles);
  f.o_part = nullptr;
  f.lse_part = nullptr;
  f.cu_q = nullptr;
  f.cu_k = nullptr;
  f.total_q = 0;
  f.total_k = 0;
  clear_paged(f);
  f.sched = nullptr;
  f.c = 0.0f;
  f.v_scale = 1.0f;
  f.idesc_qk = 0;
  f.idesc_pv = 0;
  f.wait_limit_ns = kWaitLimitNs;
  bq.lse = lse;
  bq.delta = delta;
  bq.dq = static_cast<uint16_t*>(dq);
  bq.dk = static_cast<uint16_t*>(dk);
  bq.dv = static_cast<uint16_t*>(dv);
  bq.c2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  bq.scale = scale;
  bq.n_ktiles = (Sk + kBK - 1) / kBK;
  BwdParams bk = bq;
  bk.f.total_units = static_cast<int>(static_cast<int64_t>(B) * H * bq.n_ktiles);
  bk.f.n_qtiles = (Sq + kBQKv - 1) / kBQKv;  // the dK/dV kernel steps through the queries 64 at a time
  if (D == 64)
    return causal ? launch_bwd<64, true>(dev, 0, mq, mdo, mq64, mdo64, mk, mv, mk64, mv64, bq, bk, s)
                  : launch_bwd<64, false>(dev, 1, mq, mdo, mq64, mdo64, mk, mv, mk64, mv64, bq, bk, s);
  return causal ? launch_bwd<128, true>(dev, 2, mq, mdo, mq64, mdo64, mk, mv, mk64, mv64, bq, bk, s)
                : launch_bwd<128, false>(dev, 3, mq, mdo, mq64, mdo64, mk, mv, mk64, mv64, bq, bk, s);
}
