// internal.h -- declarations shared by the translation units of libattn_gb300.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace attn {

constexpr int kHeadDim = 128;   // the only head_dim the kernels are built for
constexpr int kPageSize = 16;   // the only KV block size the kernels are built for
// The prologue stages whole tokens (all their q, k and v rows) in shared memory.
constexpr int kMaxPrologueRowsPerToken = 192;

// Device error word bits (set by kernels, read by attn_get_device_error).
enum DeviceError : int {
    kDevErrTimeout = 1,        // a bounded mbarrier wait gave up
    kDevErrBadBlockId = 2,     // a block_tables entry < 0 inside a sequence's range
    kDevErrSeqTooLong = 4,     // seq_lens[n] > max_blocks_per_seq * block_size
    kDevErrTmemAlloc = 8,      // TMEM base address outside the expected range
    kDevErrSmemLayout = 16,    // dynamic shared memory base too misaligned for the tile layout
    kDevErrBadSlot = 32,       // a slot_mapping entry outside [-1, num_blocks * block_size)
    kDevErrBadLengths = 64,    // paged prefill: a chunk longer than its context (L_q > L_kv)
    kDevErrBadPosition = 128,  // prologue: a position outside [0, max_pos) of the cos/sin table
};

// Set by the kernels (atomicOr); defined in decode.cu.  Device address of the
// word on the current device, or nullptr on failure.
int* device_error_word();
// Copy the word of the current device to *out (synchronous); optionally clear it.
cudaError_t read_device_error(int* out, bool reset);

struct DecodePlan {
    int num_seqs, H_q, H_kv, max_blocks_per_seq;
    int group;           // H_q / H_kv
    int heads_per_cta;   // query heads one CTA processes against each loaded KV page
    int chunks;          // ceil(group / heads_per_cta)
    int pages_per_split; // KV pages per split (one CTA each)
    int n_split;         // ceil(max_blocks_per_seq / pages_per_split)
    size_t o_part_bytes, lse_part_bytes;
};

DecodePlan make_decode_plan(int num_seqs, int H_q, int H_kv, int max_blocks_per_seq,
                            int pages_per_split);
size_t decode_workspace_bytes(const DecodePlan& p);

// Launch split-K main kernel + combine.  `ws` holds at least decode_workspace_bytes(p).
cudaError_t launch_decode(const DecodePlan& p, const void* q, const void* k_cache,
                          const void* v_cache, void* out, const int* block_tables,
                          const int* seq_lens, void* ws, cudaStream_t stream);

// Merge R rows of n_split partials (O normalised per split, lse natural log).
// Write num_tokens new K/V rows ([num_tokens, H_kv, 128] each) into their
// paged slots: slot s -> block s / 16, position s % 16; s == -1 is skipped.
cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const long long* slot_mapping, int num_tokens, int H_kv,
                             long long num_blocks, cudaStream_t stream);

cudaError_t launch_lse_combine(const float* O_part, const float* lse_part, void* out, int R,
                               int n_split, cudaStream_t stream);

// Process-unique id of the CUDA context current on this thread (the driver
// never hands the same id to two contexts of one process, so a context that
// replaced an earlier one, e.g. after cudaDeviceReset, is told apart from it).
// If no context is current on the thread yet, the current device's primary
// context is made current first.  Defined in api.cu.
cudaError_t current_context_id(unsigned long long* id);

// Store `e` as this thread's last CUDA error (attn_last_cuda_error) and
// return ATTN_ERR_CUDA; defined in api.cu.
int record_cuda_error(cudaError_t e);

// Prefill: O = softmax(Q K^T / sqrt(D), causal) V over [B,S,H,D] tensors.
// stall_tile >= 0 (failure-detection tests only) withholds that key tile's K
// load in every CTA, so the waits on it run out and report a timeout.
cudaError_t launch_prefill(const void* Q, const void* K, const void* V, void* O, int B, int S,
                           int H_q, int H_kv, int causal, int stall_tile, cudaStream_t stream);

// The query prologue folded into the paged prefill: per-head RMSNorm weight
// (nullptr = none), the cos/sin table of launch_rope_table with max_pos
// positions, and eps.
struct QueryPrologue {
    const void* q_weight;
    const float* cos_sin;
    int max_pos;
    float eps;
};

// Prefill of packed query chunks ([total_q, H_q, 128], cu_seqlens_q [B+1])
// against a paged cache ([num_blocks, H_kv, 16, 128]) holding seq_lens_kv[b]
// keys per sequence; query i of sequence b sits at position
// seq_lens_kv[b] - L_q(b) + i.  With qp, each query row is first normalised
// and rotated at that position (Q itself is only read).
cudaError_t launch_prefill_paged(const void* Q, const void* k_cache, const void* v_cache, void* O,
                                 const int* cu_seqlens_q, const int* seq_lens_kv,
                                 const int* block_tables, int B, int max_seqlen_q, int total_q,
                                 int H_q, int H_kv, int max_blocks_per_seq, long long num_blocks,
                                 int causal, const QueryPrologue* qp, cudaStream_t stream);

// The rotary table: per position 32 float4, entry p*32 + i*8 + m holding
// {cos a, cos b, sin a, sin b} of the angles p * base^(-2j/128) of pairs
// a = 8m + 2i and b = a + 1; computed in FP64, rounded to FP32.
cudaError_t launch_rope_table(float* cos_sin, int max_pos, double base, cudaStream_t stream);

// Per-head RMSNorm (weights q_w / k_w, nullptr = none) then NeoX RoPE of q
// [T, H_q, 128] (in place; q == nullptr: no query rows) and k [T, H_kv, 128].
// Without k_cache, k goes to k_out (may equal k); with k_cache, k and v go to
// the paged slots of slot_mapping (-1 skipped) and k_out is unused.
cudaError_t launch_qk_norm_rope(void* q, const void* k, const void* v, void* k_out,
                                const void* q_w, const void* k_w, const float* cos_sin,
                                int max_pos, const int* positions, const long long* slot_mapping,
                                void* k_cache, void* v_cache, long long num_blocks, int T,
                                int H_q, int H_kv, float eps, cudaStream_t stream);

}  // namespace attn
