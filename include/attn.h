/*
 * attn.h — C ABI of the GB300 (sm_103a) exact fused attention forward.
 *
 * The operation is dense exact attention with a per-row log-sum-exp:
 *
 *   O[b,h,i,:] = sum_j softmax_j( scale * <Q[b,h,i,:], K[b,h,j,:]> + mask[b,i,j] ) * V[b,h,j,:]
 *   LSE[b,h,i] = ln sum_{j valid} exp( scale * <Q[b,h,i,:], K[b,h,j,:]> )
 *
 * as defined in "Kernel Fusion and the Memory Wall" (thegustafson.com), section
 * "FlashAttention: avoid the full score matrix" (softmax(QK^T/sqrt(d))V, with
 * the caller's `scale` in place of 1/sqrt(d)); the softmax is the stable,
 * whole-row one of section "Softmax needs a global row statistic".  It is
 * computed tile by tile with the online max/sum correction of "Attention
 * softmax fusion" (roadmapper-2x4.pages.dev), section "The tile loop", so the
 * Sq x Sk score and probability matrices never exist in device memory.
 *
 * The mask takes only the values 0 and -inf:
 *   - key j is valid for query row i iff  j < kv_len[b]  and  (!causal || j <= i);
 *     the causal mask is top-left aligned for any Sq, Sk;
 *   - a row with no valid key (e.g. kv_len[b] == 0) yields O = +0.0 in every
 *     column and LSE = -inf, never NaN ("Attention softmax fusion", section
 *     "Things that break"; "Kernel Fusion and the Memory Wall", the paragraph on
 *     causal kernels after "A small executable reference").
 *
 * All entry points are host functions; device pointers are plain CUDA device
 * (or managed) addresses on the CURRENT device.  The caller allocates and owns
 * every buffer (including the split-KV workspace).  The library allocates no
 * device memory: its only device state is one status word and the fixed
 * scratch of attn_fwd_splitkv_noalloc, static __device__ variables that exist
 * once in every CUDA context that loads the library.
 */
#ifndef EXACT_ATTENTION_86_GB300_ATTN_H
#define EXACT_ATTENTION_86_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st* attn_stream_t;

typedef enum attn_status {
  ATTN_OK = 0,
  ATTN_ERR_NULLPTR = 1,            /* a required pointer is NULL                         */
  ATTN_ERR_ALIGN = 2,              /* q/k/v/o not 16-byte aligned, lse/kv_lens not 4-byte */
  ATTN_ERR_SHAPE = 3,              /* negative or too large B/H/Sq/Sk                   */
  ATTN_ERR_UNSUPPORTED_D = 4,      /* D is not 64 or 128                                */
  ATTN_ERR_SCALE = 5,              /* scale is NaN or infinite                          */
  ATTN_ERR_CUDA = 6,               /* a CUDA runtime/driver call failed                 */
  ATTN_ERR_DEVICE_TIMEOUT = 7,     /* a kernel wait gave up (see attn_check_device_status) */
  ATTN_ERR_UNSUPPORTED_DEVICE = 8, /* the current device is not sm_103 (GB300)          */
  ATTN_ERR_WORKSPACE = 9           /* workspace smaller than the size the call needs     */
} attn_status;

/*
 * attn_fwd — fused attention forward, asynchronous on `stream`.
 *
 * q       bf16 [B, H, Sq, D], contiguous (D innermost), device, 16-byte aligned.
 * k, v    bf16 [B, H, Sk, D], contiguous, device, 16-byte aligned.
 * o       bf16 [B, H, Sq, D], contiguous, device, 16-byte aligned; written.
 * lse     fp32 [B, H, Sq], contiguous, device, 4-byte aligned; written
 *         (natural log over the scaled scores; -inf on rows with no valid key).
 * B, H    batch and heads, >= 0.  Sq, Sk: query and key lengths, >= 0.
 *         B*H*max(Sq,Sk)*D must stay below 2^31 elements per tensor dimension
 *         set the TMA descriptor can address (checked: ATTN_ERR_SHAPE).
 * D       head dimension: 64 or 128 (else ATTN_ERR_UNSUPPORTED_D).
 * scale   multiplier of QK^T, any finite value (usually 1/sqrt(D)).
 * causal  0 or non-zero.
 * kv_lens NULL (every sequence has Sk keys) or device int32 [B]; entries are
 *         clamped to [0, Sk].  Key/value rows past kv_lens[b] that fall in the
 *         last 128-key tile are read and given weight zero, so they must hold
 *         finite values (0 * Inf would be NaN).
 *
 * Sq == 0, B == 0 or H == 0: nothing to compute, returns ATTN_OK without a
 * launch.  Sk == 0: every row has no valid key (O = 0, LSE = -inf).
 *
 * Errors: argument errors return before anything is launched.  A failed
 * launch returns ATTN_ERR_CUDA.  The call never synchronises; a device-side
 * wait that gave up (a kernel bug, never expected) is reported later by
 * attn_check_device_status.  q/k/v must not overlap o/lse.
 */
attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Sq,
                     int Sk, int D, float scale, int causal, const int32_t* kv_lens, attn_stream_t stream);

/*
 * attn_fwd_variant — attn_fwd with the kernel chosen by the caller instead of
 * by attn_fwd_kernel_choice.  Same arguments, checks, results and errors as
 * attn_fwd, plus `kernel`:
 *   ATTN_KERNEL_AUTO (-1)     the kernel attn_fwd would run;
 *   ATTN_KERNEL_ONE_TILE (0)  work units of 128 query rows;
 *   ATTN_KERNEL_TWO_TILE (1)  work units of two 128-row query tiles that share
 *                             every K/V tile (causal batches: dealt to the
 *                             SMs by a static longest-first schedule when
 *                             they have at most 4096 such units).
 * Both kernels compute the same function within the forward's tolerance;
 * they split a row's sums differently over threads, so their results are not
 * bit-identical to each other.
 * Any other `kernel` value: ATTN_ERR_SHAPE.
 */
enum { ATTN_KERNEL_AUTO = -1, ATTN_KERNEL_ONE_TILE = 0, ATTN_KERNEL_TWO_TILE = 1 };
attn_status attn_fwd_variant(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Sq,
                             int Sk, int D, float scale, int causal, const int32_t* kv_lens, int kernel,
                             attn_stream_t stream);

/*
 * attn_fwd_fp8 — the forward with FP8 (E4M3) inputs and both products on the
 * tensor cores' 8-bit path ("Fused Multi-Head Attention", the "Quantization"
 * item of the techniques fused attention combines with: FP8 data for the
 * GEMMs; "Kernel Fusion and the Memory Wall", the paragraph after "A small
 * executable reference", on FlashAttention-3's low-precision facilities).
 *
 * q       E4M3 codes [B, H, Sq, D], contiguous, device, 16-byte aligned.
 * k       E4M3 codes [B, H, Sk, D], contiguous, device, 16-byte aligned.
 * v_t     E4M3 codes of V TRANSPOSED, [B, H, D, Sk] (keys innermost), so that
 *         both operands of both products are K-major; 16-byte aligned.
 * q_descale, k_descale, v_descale: the value of a code is descale * E4M3(code)
 *         (OCP E4M3: bias 7, subnormals, no infinities, 0x7F/0xFF NaN).
 * o, lse  as attn_fwd (bf16 O, fp32 natural-log LSE over the scaled scores).
 * D 64 or 128 (else ATTN_ERR_UNSUPPORTED_D); Sk a multiple of 16 (the
 * V^T rows are Sk bytes long; else ATTN_ERR_SHAPE); scale and the descales
 * finite (else ATTN_ERR_SCALE).  Other arguments and all mask semantics as
 * attn_fwd.  The probabilities are rounded to E4M3 (scaled by 2^4, never
 * above 2^8.5) before the P V product; O and the row sums are accumulated in
 * fp32.
 */
attn_status attn_fwd_fp8(const void* q, const void* k, const void* v_t, void* o, float* lse, int B, int H, int Sq,
                         int Sk, int D, float scale, int causal, const int32_t* kv_lens, float q_descale,
                         float k_descale, float v_descale, attn_stream_t stream);

/* Layout of the E4M3 V operand of attn_fwd_fp8_ex. */
typedef enum attn_v_layout {
  ATTN_V_ROWS = 0,       /* [B, H, Sk, D], like q and k (D innermost)          */
  ATTN_V_TRANSPOSED = 1  /* [B, H, D, Sk] (keys innermost), as attn_fwd_fp8    */
} attn_v_layout;

/*
 * attn_fwd_fp8_ex — attn_fwd_fp8 with the layout of V chosen by `v_layout`.
 * With ATTN_V_ROWS, v holds E4M3 codes [B, H, Sk, D] (contiguous, 16-byte
 * aligned), the layout q and k have, and the P V product reads each V tile
 * MN-major straight from the tile the copy engine loaded; no transposition
 * is needed anywhere and Sk may have any value.  With ATTN_V_TRANSPOSED the
 * call is exactly attn_fwd_fp8 (v = V^T, Sk a multiple of 16).  Both layouts
 * give bit-identical results: the products see the same values in the same
 * order.  Any other v_layout: ATTN_ERR_SHAPE.
 */
attn_status attn_fwd_fp8_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Sq,
                            int Sk, int D, float scale, int causal, const int32_t* kv_lens, float q_descale,
                            float k_descale, float v_descale, int v_layout, attn_stream_t stream);

/*
 * attn_fwd_fp8_variant — attn_fwd_fp8_ex with the kernel chosen by the
 * caller: `kernel` as in attn_fwd_variant (ATTN_KERNEL_AUTO: the kernel
 * attn_fwd_fp8_ex runs, which attn_fwd_fp8_kernel_choice names; ATTN_KERNEL_ONE_TILE
 * or ATTN_KERNEL_TWO_TILE forced).  Both compute the same function within the
 * E4M3 forward's tolerance; they are not bit-identical to each other (their
 * row sums split differently over threads).  Any other `kernel`:
 * ATTN_ERR_SHAPE.  Everything else as attn_fwd_fp8_ex.
 */
attn_status attn_fwd_fp8_variant(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                 int Sq, int Sk, int D, float scale, int causal, const int32_t* kv_lens,
                                 float q_descale, float k_descale, float v_descale, int v_layout, int kernel,
                                 attn_stream_t stream);

/*
 * attn_fwd_varlen — the same forward over a packed batch of variable-length
 * sequences (the ragged tensors of continuous batching, "Fused Multi-Head
 * Attention", section on continuous batching): no padding is stored or read.
 *
 * q, o         bf16 [total_q, H, D], contiguous, device, 16-byte aligned.
 * k, v         bf16 [total_k, H, D], contiguous, device, 16-byte aligned.
 * lse          fp32 [H, total_q], device, 4-byte aligned.
 * cu_seqlens_q device int32 [batch + 1]: sequence b owns query tokens
 *              [cu_seqlens_q[b], cu_seqlens_q[b+1]); cu_seqlens_k likewise for
 *              keys and values.  Entries are clamped to [0, total] and to be
 *              non-decreasing, so any content keeps every access in bounds.
 * max_seqlen_q host upper bound of the query lengths (it sizes the launch).
 *              Rows of a longer sequence are computed up to the end of the
 *              work unit that holds row max_seqlen_q - 1 (units of 128 rows
 *              on the one-tile kernel, 256 on the two-tile kernel); its later
 *              rows of o and lse are left as they were.
 * Per sequence the operation is exactly attn_fwd's (causal masking top-left
 * within the sequence; a sequence with no key gives O = 0, LSE = -inf).  The
 * last 128-key tile of a sequence also reads the next sequence's first keys
 * with weight zero (they must be finite); past total_k the tile reads zeros.
 * tile_counter NULL (work is dealt round-robin to the SMs) or device uint32
 *              [2], 8-byte aligned, both zero on entry: the SMs then claim
 *              the units of work one by one, which balances ragged batches.
 *              With max_seqlen_q > 128 the call runs the two-tile kernel
 *              (units of 256 query rows of one sequence and head, claimed
 *              when the counter is given, causal or not); otherwise the
 *              one-tile kernel (units of 128 rows), which claims only for
 *              non-causal calls.  A launch leaves both words zero when it
 *              ends, so one counter serves consecutive calls on a stream;
 *              calls that share a counter must not overlap on the GPU.
 * Asynchronous on `stream`; argument errors return before any launch.
 */
attn_status attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch, int max_seqlen_q,
                            int total_q, int total_k, int H, int D, float scale, int causal, uint32_t* tile_counter,
                            attn_stream_t stream);

/*
 * attn_fwd_varlen_variant — attn_fwd_varlen with the kernel chosen by the
 * caller: `kernel` as in attn_fwd_variant (ATTN_KERNEL_AUTO: the kernel
 * attn_fwd_varlen runs: the two-tile kernel when max_seqlen_q > 128, else
 * the one-tile kernel; ATTN_KERNEL_TWO_TILE: units of two query tiles of one
 * (sequence, head), claimed from tile_counter when it is given, causal or
 * not, else dealt round-robin).  Both compute the
 * same function within the forward's tolerance; they are not bit-identical
 * to each other.  Any other `kernel`: ATTN_ERR_SHAPE.  Everything else as
 * attn_fwd_varlen.
 */
attn_status attn_fwd_varlen_variant(const void* q, const void* k, const void* v, void* o, float* lse,
                                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch,
                                    int max_seqlen_q, int total_q, int total_k, int H, int D, float scale, int causal,
                                    uint32_t* tile_counter, int kernel, attn_stream_t stream);

/*
 * attn_fwd_paged — the packed-query forward with keys and values read through
 * a page table from a paged KV cache (the PagedAttention layout named in
 * "Fused Multi-Head Attention", section on continuous batching): a sequence's
 * keys need not be contiguous in memory.
 *
 * q, o         bf16 [total_q, H, D] packed queries, as in attn_fwd_varlen.
 * lse          fp32 [H, total_q].
 * cu_seqlens_q device int32 [batch + 1] query offsets, as in attn_fwd_varlen.
 * k_cache,     bf16 [num_pages, page_size, H, D], contiguous, device, 16-byte
 * v_cache      aligned.
 * seqlens_k    device int32 [batch]: keys of sequence b, clamped to
 *              [0, max_pages_per_seq * page_size].
 * block_table  device int32 [batch, max_pages_per_seq]: key j of sequence b is
 *              slot j % page_size of page block_table[b][j / page_size]
 *              (entries clamped to [0, num_pages - 1]; entries past the
 *              sequence's last key are never read).
 * page_size    a multiple of 64 (each 64-key half of a 128-key tile is one copy).
 * Per sequence the operation is attn_fwd's on its gathered keys (causal:
 * query i of the sequence sees keys j <= i).  Slots of the last used page past
 * seqlens_k[b] that share a 64-key half with a valid key are read with weight
 * zero and must hold finite values; whole halves past it read zeros.
 * tile_counter as attn_fwd_varlen.  Asynchronous on `stream`; argument errors
 * return before any launch (page_size, num_pages or max_pages_per_seq out of
 * range: ATTN_ERR_SHAPE).
 */
attn_status attn_fwd_paged(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                           const int32_t* cu_seqlens_q, const int32_t* seqlens_k, const int32_t* block_table,
                           int batch, int max_seqlen_q, int total_q, int num_pages, int page_size,
                           int max_pages_per_seq, int H, int D, float scale, int causal, uint32_t* tile_counter,
                           attn_stream_t stream);

/*
 * attn_fwd_paged_variant — attn_fwd_paged with the kernel chosen by the
 * caller: `kernel` as in attn_fwd_varlen_variant (ATTN_KERNEL_AUTO: the
 * kernel attn_fwd_paged runs, the two-tile kernel when max_seqlen_q > 128,
 * else the one-tile kernel; ATTN_KERNEL_TWO_TILE: units of two query tiles
 * of one (sequence, head), claimed from tile_counter when it is given, else
 * dealt round-robin).  Any other
 * `kernel`: ATTN_ERR_SHAPE.  Everything else as attn_fwd_paged.
 */
attn_status attn_fwd_paged_variant(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                                   const int32_t* cu_seqlens_q, const int32_t* seqlens_k,
                                   const int32_t* block_table, int batch, int max_seqlen_q, int total_q,
                                   int num_pages, int page_size, int max_pages_per_seq, int H, int D, float scale,
                                   int causal, uint32_t* tile_counter, int kernel, attn_stream_t stream);

/*
 * attn_fwd_splitkv — the same forward with the keys of every (b, h, 128-row
 * query block) cut into `num_splits` contiguous ranges of 128-key tiles that
 * run as separate units of work, then merged (split-KV).  It raises the
 * parallelism of shapes with few query blocks (short Sq, few heads, decode)
 * at the cost of a workspace and one merge pass.
 *
 * Each range produces the normalised partial output O_s = sum p_j v_j / sum p_j
 * and LSE_s over its keys (the tile loop of "Attention softmax fusion",
 * section "The tile loop", run on the range); the merge applies the running
 * max / normaliser correction once per range (see attn_lse_merge).
 *
 * Arguments as attn_fwd, plus:
 * num_splits       1 .. 128.  Ranges are whole tiles, so a range may be empty;
 *                  an empty range contributes nothing.
 * workspace        device memory, 256-byte aligned, caller-owned, at least
 *                  attn_fwd_splitkv_workspace_size(B, H, Sq, D, num_splits)
 *                  bytes (else ATTN_ERR_WORKSPACE).  Its contents on entry are
 *                  irrelevant; the call overwrites it.  Calls that use one
 *                  workspace must not overlap on the GPU.
 * Two kernels are launched on `stream`; the call never synchronises.
 */
size_t attn_fwd_splitkv_workspace_size(int B, int H, int Sq, int D, int num_splits);

/*
 * attn_fwd_splitkv_suggest_splits — a key-range count for attn_fwd_splitkv on
 * a GPU with `num_sms` SMs.  With U = B * H * ceil(Sq / 128) units of work, at
 * most S_max = num_sms / U ranges (capped by the number of 128-key tiles and
 * by 128) keep the units within one wave of SMs; the result is the largest
 * S <= S_max that cuts the tiles into equal ranges, unless that is below
 * S_max / 2 (then S_max).  Returns 1 when U >= num_sms (splitting gains
 * nothing) or when a size is 0, and 0 for a negative size or num_sms < 1.
 * Host arithmetic only: no CUDA call, no device needed.
 */
int attn_fwd_splitkv_suggest_splits(int B, int H, int Sq, int Sk, int num_sms);

attn_status attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Sq,
                             int Sk, int D, float scale, int causal, const int32_t* kv_lens, int num_splits,
                             void* workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_fwd_splitkv_noalloc — attn_fwd_splitkv for callers that cannot
 * allocate device memory and have no workspace to hand over: a plugin inside
 * a host framework that owns every byte of device memory and gives its
 * plugins none, a serving loop that runs under a fixed memory budget, or code
 * that must never call cudaMalloc / cudaFree because those calls may
 * synchronise the device.  The partial results go to a fixed scratch array of
 * ATTN_SPLITKV_SCRATCH_BYTES bytes inside the library (a static __device__
 * array).  That array is part of the library's device image: every CUDA
 * context that loads the library reserves ATTN_SPLITKV_SCRATCH_BYTES of
 * device memory for it until the context ends, whether or not this entry
 * point is ever called.  In host code the array's name is not a device
 * address; each call looks the address up in the current context
 * (cudaGetSymbolAddress, which allocates nothing).  The first call in a
 * context may be the one that loads the library's module there, so make it
 * before any stream capture.
 *
 * Arguments as attn_fwd_splitkv minus the workspace.  A call whose
 * attn_fwd_splitkv_workspace_size(B, H, Sq, D, num_splits) exceeds the
 * scratch returns ATTN_ERR_WORKSPACE before any CUDA call.  The call makes no
 * cudaMalloc, cudaFree or other allocating call.  Every call in one context
 * shares the scratch, and the scratch keeps what the last call wrote (every
 * element a call reads back was written by that same call, so no clearing is
 * needed): calls that overlap on the GPU race on it, so issue them on one
 * stream or order them with events.
 */
#define ATTN_SPLITKV_SCRATCH_BYTES (32u << 20)

attn_status attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                     int Sq, int Sk, int D, float scale, int causal, const int32_t* kv_lens,
                                     int num_splits, attn_stream_t stream);

/*
 * attn_lse_merge — combine attention results computed over disjoint key sets
 * into the result over their union ("Kernel Fusion and the Memory Wall",
 * section "FlashAttention: avoid the full score matrix": rescale each part by
 * exp(m - m') so that all share one denominator; here m is each part's LSE):
 *
 *   M = max_s LSE_s,  w_s = exp(LSE_s - M),  O = sum_s w_s O_s / sum_s w_s,
 *   LSE = M + ln sum_s w_s;   every LSE_s = -inf  ->  O = +0.0, LSE = -inf.
 *
 * o_parts    fp32 [num_parts][rows][D] normalised partial outputs, device, 16-B aligned.
 * lse_parts  fp32 [num_parts][rows] partial LSE (natural log), device, 4-B aligned.
 * o          bf16 [rows][D] output, device, 8-B aligned.   lse: fp32 [rows] output.
 * rows >= 0, num_parts >= 1, D in {64, 128}.  Asynchronous on `stream`.
 * This is the exchange step a key-sharded (context-parallel) forward needs.
 */
attn_status attn_lse_merge(const float* o_parts, const float* lse_parts, int num_parts, void* o, float* lse,
                           long long rows, int D, attn_stream_t stream);

/*
 * attn_bwd — gradients of attn_fwd's O with respect to Q, K and V for an
 * upstream gradient dO (the LSE output is not differentiated).  The pages
 * give the forward only ("Fused Multi-Head Attention" notes that fused
 * kernels also make training with long sequences efficient); the gradients
 * are the chain rule on the softmax: with P = exp(scale QK^T + mask - LSE),
 *   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - Delta),  Delta_i = <dO_i, O_i>,
 *   dQ = scale dS K,  dK = scale dS^T Q.
 *
 * q, k, v, o, lse  the forward's inputs and outputs (layouts as attn_fwd).
 * dout             bf16 [B, H, Sq, D], contiguous, device, 16-byte aligned.
 * dq               bf16 [B, H, Sq, D] output; dk, dv: bf16 [B, H, Sk, D].
 * workspace        device, 256-byte aligned, caller-owned, at least
 *                  attn_bwd_workspace_size(B, H, Sq) bytes (fp32 Delta).
 * Other arguments, masks and the D restriction as attn_fwd.  Rows without a
 * valid key get dQ = 0; keys no query sees (past kv_lens, or masked for
 * every query) get dK = dV = 0.  Sq == 0: dK = dV = 0; Sk == 0: dQ = 0.
 * Three kernels on `stream` (Delta, dQ, dK/dV); the call never synchronises.
 */
size_t attn_bwd_workspace_size(int B, int H, int Sq);

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                     void* dq, void* dk, void* dv, int B, int H, int Sq, int Sk, int D, float scale, int causal,
                     const int32_t* kv_lens, void* workspace, size_t workspace_bytes, attn_stream_t stream);

/* Static, human-readable description of a status code. */
const char* attn_get_error_string(attn_status status);

/*
 * attn_check_device_status — synchronises `stream`, then reads and clears the
 * current device's status word.  Returns ATTN_ERR_DEVICE_TIMEOUT if any kernel
 * of this library gave up on a bounded wait since the last check (the kernel
 * then skipped the rest of its work and released its resources), ATTN_ERR_CUDA
 * if the synchronisation failed, else ATTN_OK.  If `site` is not NULL it
 * receives the code of the first wait that gave up (0 if none).
 */
attn_status attn_check_device_status(attn_stream_t stream, uint32_t* site);

/*
 * attn_selftest_wait_timeout — failure-detection self test.  Launches one
 * 32-thread block that waits on a shared-memory mbarrier that nothing ever
 * arrives on, with the same bounded wait the attention kernel uses but a limit
 * of `limit_ns` nanoseconds (1 .. 2e9).  The wait gives up, sets the status
 * word and the block exits normally; attn_check_device_status then returns
 * ATTN_ERR_DEVICE_TIMEOUT.  No fault, trap or unbounded spin is involved.
 */
attn_status attn_selftest_wait_timeout(int64_t limit_ns, attn_stream_t stream);

/*
 * attn_selftest_fwd_abort — failure-detection self test of the attention
 * kernel itself ("Attention softmax fusion", section "Things that break": a
 * fused kernel must fail without corrupting what it shares).  Runs
 * attn_fwd_variant (same arguments, same checks, `kernel` as there; Sk >= 1
 * required) with every bounded wait
 * limited to `limit_ns` nanoseconds (1000 .. 2e9) instead of 2 s, and with
 * block 0's producer leaving out its K fill number `skip_fill` (>= 0,
 * counted over that block's K tiles in its order of work).  Nothing ever
 * arrives for that fill, so a wait in block 0 gives up: the block records the
 * site, raises its abort flag, every role drains its copies and products,
 * frees Tensor Memory and returns; attn_check_device_status then reports
 * ATTN_ERR_DEVICE_TIMEOUT.  The other blocks finish their units normally
 * (unless `limit_ns` is shorter than their own legitimate waits).  If block 0
 * has fewer K fills than skip_fill + 1 nothing is left out.  The rows of
 * block 0's units are left undefined.  No fault, trap or unbounded spin is
 * involved.
 */
attn_status attn_selftest_fwd_abort(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                    int Sq, int Sk, int D, float scale, int causal, const int32_t* kv_lens,
                                    int kernel, int skip_fill, int64_t limit_ns, attn_stream_t stream);

/*
 * attn_selftest_launch_floor — measurement aid, no attention arithmetic.
 * Launches `grid` blocks (1 .. 65535) of a kernel with the attention
 * forward's launch shape for head dimension D (64 or 128): 384 threads and the
 * same dynamic shared memory, so one block per SM.  mode 0: the kernel returns
 * at once (the cost of the launch itself); mode 1: it does only the forward
 * kernel's fixed per-block set-up and tear-down (mbarrier initialisation,
 * Tensor Memory allocation of 512 columns, the block-wide synchronisations,
 * Tensor Memory release) with no loads and no products.  Timing it against
 * the forward on a small workload separates the launch and set-up floor from
 * the work ("Attention softmax fusion", section "Things that break", warns
 * against judging a fused kernel by one short sequence length).
 * Errors: ATTN_ERR_SHAPE for a grid or mode out of range,
 * ATTN_ERR_UNSUPPORTED_D, ATTN_ERR_CUDA / ATTN_ERR_UNSUPPORTED_DEVICE as for
 * the other calls.  Asynchronous on `stream`.
 */
attn_status attn_selftest_launch_floor(int grid, int D, int mode, attn_stream_t stream);

/*
 * attn_fwd_kernel_choice — which kernel attn_fwd runs for a padded bf16 batch
 * of B x H heads of Sq queries and Sk keys, head dimension D, causal or not,
 * on a device with `num_sms` SMs.  Returns 1 for the two-query-tile kernel
 * (units of 256 query rows), 0 for the one-tile kernel (units of 128 rows),
 * -1 for a negative argument or D other than 64 and 128.  The two compute
 * the same function; the choice is a cost model of the work units
 * (non-causal: waves of equal units over the SMs; causal: the larger of the
 * longest unit and the mean work per SM, with at most 4096 two-tile units)
 * and never depends on the data.  At D = 64 the products take half the
 * D = 128 time, so the softmax, which the two-tile kernel interleaves, weighs
 * more and that kernel is chosen more often.  Host only: no CUDA call.
 */
int attn_fwd_kernel_choice(int B, int H, int Sq, int Sk, int D, int causal, int num_sms);

/*
 * attn_fwd_fp8_kernel_choice — the same for attn_fwd_fp8_ex (E4M3 inputs),
 * whose products take half the bf16 time: the two-tile kernel is chosen as
 * for bf16 D = 64 (non-causal: a cheaper pair in the wave model; causal: from
 * 1024 queries on, within the 4096-unit limit).  Same results and errors as
 * attn_fwd_kernel_choice.
 */
int attn_fwd_fp8_kernel_choice(int B, int H, int Sq, int Sk, int D, int causal, int num_sms);

/*
 * attn_fwd_pair_schedule — the static deal of a causal batch's two-tile units
 * that attn_fwd uses on the two-tile kernel: owner[t] (host memory, at least
 * max_units bytes, caller-owned) receives the block that runs unit t, t in
 * the kernel's unit order: groups of `head_group` (b, h) heads in b-major
 * order, within a group the 256-row query pairs from the last one down, each
 * over the group's heads.  Each unit in turn goes to the block with the least
 * modelled work so far (lowest index among equals); the model counts a unit's
 * key tiles ("Attention softmax fusion", section "The tile loop": one key
 * tile per step) plus a fixed part.  Returns the number of units
 * (B * H * ceil(Sq / 256)), or -1 when that exceeds max_units, grid is not
 * 1 .. 256, head_group < 1 or an argument is negative.  Host only.
 */
int64_t attn_fwd_pair_schedule(int B, int H, int Sq, int Sk, int head_group, int grid, uint8_t* owner,
                               int64_t max_units);

/* ABI version of this header (incremented on any signature change). */
int attn_abi_version(void);

#define ATTN_ABI_VERSION 18

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTENTION_86_GB300_ATTN_H */
