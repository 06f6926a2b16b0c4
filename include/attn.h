/*
 * attn.h -- C ABI of libattn_gb300: grouped-query attention for one GB300
 * (sm_103a) GPU.  Plain pointers and sizes only.
 *
 * Conventions for every entry point
 *  - Tensors are caller-owned DEVICE buffers, dense and contiguous in the
 *    layouts stated below (no stride arguments).  FP16 buffers must be
 *    16-byte aligned; int32 buffers 4-byte aligned.
 *  - Calls are asynchronous on `stream` (0 = the legacy default stream of the
 *    current device) and return once the kernels are launched.  They never
 *    synchronise the device, never print, never exit.
 *  - Arguments are validated on the host before anything is launched; on any
 *    non-zero return nothing was launched (except ATTN_ERR_CUDA from the
 *    launch itself).
 *  - Return 0 (ATTN_OK) on success, else a negative ATTN_ERR_* code.
 *  - Preconditions the host cannot check (the library never reads device
 *    memory on the host) are listed per call.  The kernels check the cheap
 *    ones on the device, skip the offending work and record it in the device
 *    error word (attn_get_device_error).
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = -1,  /* null/misaligned pointer, negative size, H_q % H_kv != 0, O aliasing an input */
    ATTN_ERR_UNSUPPORTED = -2,  /* head_dim != 128 or block_size != 16 */
    ATTN_ERR_CUDA = -3,         /* a CUDA runtime call failed; see attn_last_cuda_error() */
    ATTN_ERR_TIMEOUT = -4,      /* device error word: a bounded on-chip wait gave up */
    ATTN_ERR_BAD_INPUT = -5,    /* device error word: negative block id, seq_len beyond the table, slot out of range */
    ATTN_ERR_WORKSPACE = -6     /* caller workspace missing or smaller than required */
};

/*
 * Prefill attention.
 * Operation: "Tutorial: Adding a New Kernel to RL.cu" (add-cuda-kernel page),
 * include/kernels/attention.cuh, "Flash Attention 2 -- Prefill":
 *   O[b,i,h,:] = sum_j softmax_j(Q[b,i,h,:].K[b,j,g,:] / sqrt(D)) V[b,j,g,:]
 *   with g = h*H_kv/H_q, j over 0..i if causal, else over 0..S-1.
 * Q, O : [B, S, H_q, D] FP16.   K, V : [B, S, H_kv, D] FP16.
 * D must be 128 (else ATTN_ERR_UNSUPPORTED); H_q % H_kv == 0.
 * B == 0 or S == 0 is a no-op.  O must not overlap Q, K or V.
 * Accumulation is FP32; the output is rounded to nearest-even FP16.
 */
ATTN_API int attn_prefill(const void* Q, const void* K, const void* V, void* O, int B, int S,
                          int H_q, int H_kv, int D, int causal, cudaStream_t stream);

/*
 * Prefill of new query chunks against a paged KV cache (variable lengths,
 * cached prefix): the chunked-prefill step that combines the prefill of
 * "Flash Attention 2 -- Prefill" with the cache layout of "Paged Attention --
 * Decode" (same header).  Sequence b contributes L_q = cu_seqlens_q[b+1] -
 * cu_seqlens_q[b] queries, packed at rows cu_seqlens_q[b].. of Q and O; its
 * context holds L_kv = seq_lens_kv[b] keys in the cache, the last L_q of them
 * belonging to the chunk itself (its K/V appended already), so L_q <= L_kv.
 * Query i sits at position L_kv - L_q + i; with causal != 0 it attends to
 * keys 0..L_kv-L_q+i, else to all L_kv keys; scale 1/sqrt(D), g = h*H_kv/H_q.
 * Q, O         : [total_q, H_q, D] FP16, total_q = cu_seqlens_q[B]
 * k/v_cache    : [num_blocks, H_kv, block_size, D] FP16
 * cu_seqlens_q : [B+1] int32 (0 first, non-decreasing); seq_lens_kv : [B] int32
 * block_tables : [B, max_blocks_per_seq] int32
 * max_seqlen_q : an upper bound of every L_q (sizes the launch).
 * D must be 128 and block_size 16.  B, total_q or max_seqlen_q == 0 is a no-op.
 * Cache slots past a context and table entries past its pages may hold
 * anything; a page id outside [0, num_blocks) reads as zeros.  Device-checked
 * preconditions (flagged, ATTN_ERR_BAD_INPUT): 0 <= cu_seqlens_q[b] <=
 * cu_seqlens_q[b+1] <= total_q and L_q <= L_kv (else the sequence is skipped),
 * L_q <= max_seqlen_q (else its extra rows are not computed), L_kv <=
 * max_blocks_per_seq*block_size (else clamped).
 */
ATTN_API int attn_prefill_paged(const void* Q, const void* k_cache, const void* v_cache, void* O,
                                const int* cu_seqlens_q, const int* seq_lens_kv,
                                const int* block_tables, int B, int max_seqlen_q, int total_q,
                                int H_q, int H_kv, int D, int max_blocks_per_seq, int block_size,
                                long long num_blocks, int causal, cudaStream_t stream);

/*
 * attn_prefill_paged with the query side of the attention-input prologue
 * folded into the kernel's Q load ("GRPO-CUDA Project Memory" page, "Model
 * forward pass": QK-norm -> RoPE -> KV append -> attention; "Qwen3-Specific
 * Notes" and "RoPE design" for the per-head RMSNorm and the split-half
 * rotation).  Q holds the raw query projections and is only read: query i of
 * sequence b is first normalised, y = w * x / sqrt(mean(x^2) + eps) (no norm
 * when q_weight is NULL), and rotated at its position L_kv - L_q + i with the
 * table of attn_rope_cos_sin_table (max_pos positions), in FP32 rounded once
 * to FP16 (attn_qk_norm_rope's definition; here x*w is formed exactly before
 * the 1/rms factor, so a value may differ from that call's by one FP16 ulp),
 * and then attends exactly as in attn_prefill_paged.  The cache must already hold normalised and
 * rotated keys (attn_qk_norm_rope_append with Q = NULL writes them).
 * q_weight : [D] FP16 or NULL (16-byte aligned); cos_sin : [max_pos, D] FP32
 * (16-byte aligned); eps >= 0.  A query whose position lies outside
 * [0, max_pos) is left unrotated and flagged (bit 128, ATTN_ERR_BAD_INPUT).
 * Everything else as attn_prefill_paged.  One launch.
 */
ATTN_API int attn_prefill_paged_qk_norm_rope(const void* Q, const void* k_cache, const void* v_cache,
                                             void* O, const int* cu_seqlens_q,
                                             const int* seq_lens_kv, const int* block_tables,
                                             const void* q_weight, const float* cos_sin,
                                             int max_pos, float eps, int B, int max_seqlen_q,
                                             int total_q, int H_q, int H_kv, int D,
                                             int max_blocks_per_seq, int block_size,
                                             long long num_blocks, int causal, cudaStream_t stream);

/*
 * Failure-detection test hook (not for production use): attn_prefill, except
 * that the K tile with index stall_tile (>= 0) is never loaded in any CTA
 * that reaches it.  The on-chip waits for that tile run out after their
 * ~1 s limit; every role of the kernel then leaves its loop, waits for its own
 * copies and MMAs in flight, releases tensor memory and exits, and the device
 * error word reports a timeout (attn_get_device_error -> ATTN_ERR_TIMEOUT).
 * O is left unspecified for the affected rows.  Lets a test exercise the
 * timeout path of the real kernel without faulting or hanging the GPU.
 */
ATTN_API int attn_debug_prefill_stall(const void* Q, const void* K, const void* V, void* O, int B,
                                      int S, int H_q, int H_kv, int D, int causal, int stall_tile,
                                      cudaStream_t stream);

/*
 * Single-token decode over a paged KV cache.
 * Operation: same page, "Paged Attention -- Decode":
 *   out[n,h,:] = sum_{t < seq_lens[n]} softmax_t(q[n,h,:].K_t / sqrt(D)) V_t,
 *   K_t = k_cache[block_tables[n, t/block_size], g, t % block_size, :] (V_t alike),
 *   g = h*H_kv/H_q.  seq_lens counts the context including the new token.
 * q, out        : [num_seqs, H_q, D] FP16
 * k/v_cache     : [num_blocks, H_kv, block_size, D] FP16
 * block_tables  : [num_seqs, max_blocks_per_seq] int32, logical -> physical block
 * seq_lens      : [num_seqs] int32
 * D must be 128 and block_size 16 (else ATTN_ERR_UNSUPPORTED).
 * A sequence with seq_lens[n] == 0 gets out = 0.  num_seqs == 0 is a no-op.
 * Only the first ceil(seq_lens[n]/block_size) table entries of a row and the
 * first seq_lens[n] slots of the context are read; the rest may hold anything.
 * Device-side preconditions: 0 <= block_tables[n][p] < num_blocks for the
 * pages in use (negative ids are skipped and flagged; ids >= num_blocks cannot
 * be detected: there is no num_blocks argument), and
 * seq_lens[n] <= max_blocks_per_seq*block_size (longer ones are clamped and
 * flagged).
 * Scratch for the split-K partials comes from a library-owned grow-only
 * buffer per (device, stream); growing it calls cudaMalloc/cudaFree (which
 * synchronise the device).  A buffer of a context that has been replaced
 * since (cudaDeviceReset) is forgotten and a new one allocated.  Use
 * attn_decode_paged_ws to pass your own.
 */
ATTN_API int attn_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                               void* out, const int* block_tables, const int* seq_lens,
                               int num_seqs, int H_q, int H_kv, int D, int max_blocks_per_seq,
                               int block_size, cudaStream_t stream);

/*
 * Bytes of scratch attn_decode_paged_ws needs for these sizes.
 * pages_per_split: KV pages per split-K work unit.  <= 0 picks the default: 64,
 * halved (down to 4) while the grid would hold fewer than 12 CTAs per SM of
 * the current device (1824 on a 152-SM GB300; 152 SMs are assumed when the
 * device cannot be queried).  Returns 0 for invalid sizes.
 */
ATTN_API size_t attn_decode_paged_workspace_bytes(int num_seqs, int H_q, int H_kv, int D,
                                                  int max_blocks_per_seq, int block_size,
                                                  int pages_per_split);

/*
 * attn_decode_paged with caller scratch: `workspace` is a device buffer of
 * at least attn_decode_paged_workspace_bytes(...) bytes, 256-byte aligned,
 * owned by the caller, and must not be used by another call that overlaps on
 * the GPU.  The call allocates nothing.  Same semantics otherwise; the result
 * does not depend on pages_per_split beyond FP32 rounding.
 */
ATTN_API int attn_decode_paged_ws(const void* q, const void* k_cache, const void* v_cache,
                                  void* out, const int* block_tables, const int* seq_lens,
                                  int num_seqs, int H_q, int H_kv, int D, int max_blocks_per_seq,
                                  int block_size, int pages_per_split, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream);

/*
 * attn_decode_paged for callers that cannot allocate device memory.
 * The pages have no counterpart of this call.  It is for users of this
 * library who cannot call cudaMalloc: code hosted in another runtime that
 * owns all device memory and offers no allocator, programs under a fixed
 * memory budget, and loops that must not risk the device-wide
 * synchronisation cudaMalloc/cudaFree can bring.
 * Same arguments, semantics and preconditions as attn_decode_paged.  The
 * split-K scratch is a buffer of ATTN_NOALLOC_SCRATCH_BYTES (32 MiB)
 * compiled into the library: every GPU that loads the library's device code
 * holds it until the process exits.  The call allocates nothing.
 *  - A problem whose scratch (attn_decode_paged_workspace_bytes with
 *    pages_per_split = 0) exceeds ATTN_NOALLOC_SCRATCH_BYTES is refused with
 *    ATTN_ERR_WORKSPACE before anything is launched.
 *  - The first call on a device looks up the buffer's device address with
 *    cudaGetSymbolAddress (so does the first call after the device's context
 *    was replaced, e.g. by cudaDeviceReset); make that first call before any
 *    stream capture.
 *  - Every call on a device shares the one buffer, which keeps the last
 *    call's contents.  Nothing needs clearing (each partial that is read is
 *    written earlier in the same call), but calls that overlap on the GPU
 *    (e.g. on two streams) race on it: serialise them.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
ATTN_API int attn_decode_paged_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                       void* out, const int* block_tables, const int* seq_lens,
                                       int num_seqs, int H_q, int H_kv, int D,
                                       int max_blocks_per_seq, int block_size,
                                       cudaStream_t stream);

/*
 * Append new tokens' K and V rows to the paged cache ("GRPO-CUDA Project
 * Memory" page, "KV Cache design": reshape-and-cache with
 * slot_mapping[token] = physical_block * block_size + offset, int64; slot -1
 * is a padding token and is skipped, "Known bugs fixed").
 * k_new, v_new : [num_tokens, H_kv, D] FP16
 * k/v_cache    : [num_blocks, H_kv, block_size, D] FP16, updated in place
 * slot_mapping : [num_tokens] int64 (8-byte aligned)
 * D must be 128 and block_size 16.  A slot outside [-1, num_blocks*block_size)
 * is skipped and flagged in the device error word (ATTN_ERR_BAD_INPUT).  Two
 * tokens mapped to the same slot race (the last write wins, unspecified).
 * The new rows must not overlap the caches.
 */
ATTN_API int attn_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                            const long long* slot_mapping, int num_tokens, int H_kv, int D,
                            int block_size, long long num_blocks, cudaStream_t stream);

/*
 * One decode step with its KV append: attn_kv_append of one new token per
 * sequence (k_new/v_new [num_seqs, H_kv, D], slot_mapping [num_seqs]) followed
 * on the same stream by attn_decode_paged over the updated cache (seq_lens
 * already counting the new token), as the page's layer order prescribes (KV
 * append, then attention: "Model forward pass").  Two launches in one call;
 * scratch as attn_decode_paged.
 */
ATTN_API int attn_decode_paged_append(const void* q, const void* k_new, const void* v_new,
                                      void* k_cache, void* v_cache, void* out,
                                      const long long* slot_mapping, const int* block_tables,
                                      const int* seq_lens, int num_seqs, int H_q, int H_kv, int D,
                                      int max_blocks_per_seq, int block_size, long long num_blocks,
                                      cudaStream_t stream);

/*
 * Attention-input prologue, step 1: the rotary cos/sin table.  Pair j
 * (element j with element j + D/2, j < D/2) turns by a_j(p) = p * base^(-2j/D)
 * at position p (the angle of the Kimi-K2.6 KernelBench trace, fused
 * cross-attention page); the FP32 table indexed by position is the "RoPE
 * design" of the "GRPO-CUDA Project Memory" page.  The buffer holds max_pos*D
 * floats (16-byte aligned, caller-owned): per position 512 bytes, ordered for
 * the prologue kernel's loads as float4 entries
 *   cos_sin[(p*32 + i*8 + m)*4 + 0..3] = {cos a_j, cos a_j+1, sin a_j, sin a_j+1},
 *   j = 8m + 2i,  m < 8,  i < 4.
 * The angles and their sines and cosines are computed in FP64 and rounded
 * once, so late positions lose no accuracy.  D must be 128; base > 0 (the
 * pages print no value: it is the model's RoPE base).  Build it once.
 */
ATTN_API int attn_rope_cos_sin_table(float* cos_sin, int max_pos, int D, double base,
                                     cudaStream_t stream);

/*
 * Attention-input prologue, step 2, in place: per-head QK-norm then NeoX RoPE
 * ("GRPO-CUDA Project Memory" page, "Qwen3-Specific Notes": RMSNorm over each
 * head's 128 values before RoPE, eps 1e-6 there; "RoPE design": element i
 * rotates with element i + D/2):
 *   y = w * x / sqrt(mean(x^2) + eps)              (no norm when w is NULL)
 *   x'[i] = y[i] c - y[i+64] s,  x'[i+64] = y[i+64] c + y[i] s,
 *   (c, s) = (cos, sin) of pair i at positions[t], from the table above
 * Q         : [num_tokens, H_q, D] FP16, rewritten in place
 * K         : [num_tokens, H_kv, D] FP16, rewritten in place
 * q_weight, k_weight : [D] FP16 RMSNorm weights, or NULL for RoPE only
 * cos_sin   : the table of attn_rope_cos_sin_table, max_pos positions
 * positions : [num_tokens] int32, each token's absolute position
 * FP32 arithmetic, FP16 results rounded to nearest.  D must be 128 and
 * H_q + H_kv at most 192 (ATTN_ERR_UNSUPPORTED otherwise).  A token whose
 * position lies outside [0, max_pos) is left unchanged and flagged in the
 * device error word (bit 128, ATTN_ERR_BAD_INPUT).  Q and K must not overlap
 * each other or the read-only inputs.  One launch.
 */
ATTN_API int attn_qk_norm_rope(void* Q, void* K, const void* q_weight, const void* k_weight,
                               const float* cos_sin, int max_pos, const int* positions,
                               int num_tokens, int H_q, int H_kv, int D, float eps,
                               cudaStream_t stream);

/*
 * The prologue fused with the KV append, in the page's layer order (QK-norm,
 * RoPE, KV append, then attention: "Model forward pass"): Q is normalised and
 * rotated in place as in attn_qk_norm_rope; K is normalised and rotated and V
 * copied straight into their paged cache slots (attn_kv_append's slot rules:
 * slot -1 skipped, out-of-range flagged with bit 32); K and V themselves are
 * only read.  Q may be NULL: then only keys and values are processed (the
 * queries' part runs inside attn_prefill_paged_qk_norm_rope) and H_q is not
 * used beyond its check.  Caches [num_blocks, H_kv, block_size, D] FP16,
 * block_size 16, must not overlap any input; H_q (0 when Q is NULL) + 2*H_kv
 * at most 192.  One launch.
 */
ATTN_API int attn_qk_norm_rope_append(void* Q, const void* K, const void* V, const void* q_weight,
                                      const void* k_weight, const float* cos_sin, int max_pos,
                                      const int* positions, const long long* slot_mapping,
                                      void* k_cache, void* v_cache, int num_tokens, int H_q,
                                      int H_kv, int D, int block_size, long long num_blocks,
                                      float eps, cudaStream_t stream);

/*
 * Merge partial attention results over disjoint key segments by their
 * log-sum-exp (the combine step of split-K decode):
 *   L = log sum_i exp(lse[r,i]),  out[r,:] = sum_i exp(lse[r,i] - L) O_part[r,i,:]
 * O_part : [R, n_split, D] FP32, each normalised over its segment
 * lse    : [R, n_split]    FP32 natural log; -inf marks an empty segment
 * out    : [R, D] FP16 (a row whose segments are all empty gets 0).
 * D must be 128.  Basis: the online-softmax identity o_N/l_N = sum v e^s / sum e^s
 * worked through in the Kimi-K2.6 KernelBench trace (fused cross-attention page).
 */
ATTN_API int attn_lse_combine(const float* O_part, const float* lse, void* out, int R,
                              int n_split, int D, cudaStream_t stream);

/* Free every library-owned workspace (synchronises the devices that own one). */
ATTN_API int attn_release_workspace(void);

/*
 * Read the device error word of the current device (synchronises the device).
 * *code receives the raw bits (1 timeout, 2 negative block id, 4 seq_len
 * beyond the table, 16 shared-memory layout did not fit, 32 slot out of
 * range, 64 a paged-prefill chunk longer than its context or than
 * max_seqlen_q, 128 a prologue position outside the cos/sin table); the return is ATTN_OK if it is 0, else ATTN_ERR_TIMEOUT
 * or ATTN_ERR_BAD_INPUT.  reset != 0 clears it.
 */
ATTN_API int attn_get_device_error(int* code, int reset);

/* cudaError_t value behind the last ATTN_ERR_CUDA returned on this thread. */
ATTN_API int attn_last_cuda_error(void);

/* Static description of a status code. */
ATTN_API const char* attn_status_string(int status);

/* Library version: major*10000 + minor*100 + patch. */
ATTN_API int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
