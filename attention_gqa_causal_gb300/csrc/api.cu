// api.cu -- the C ABI of libattn_gb300: argument validation, workspace
// ownership, error mapping.  Every compute step runs in the kernels of
// prefill.cu, decode.cu and rope.cu.
#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>

#include "attn.h"
#include "internal.h"

namespace {

thread_local int t_last_cuda_error = 0;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name)
{
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(p);
}

int cuda_fail(cudaError_t e)
{
    t_last_cuda_error = static_cast<int>(e);
    return ATTN_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

int check_heads(int H_q, int H_kv)
{
    if (H_q < 1 || H_kv < 1 || H_q % H_kv != 0)
        return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

// Library-owned split-K scratch: one grow-only buffer per (device, stream),
// tagged with the context it was allocated in.  A buffer from a context that
// has since been replaced (cudaDeviceReset) went away with that context: it is
// forgotten, never freed or used.
struct Workspace {
    void* ptr = nullptr;
    size_t bytes = 0;
    unsigned long long ctx = 0;
};
std::mutex g_ws_mutex;
std::map<std::pair<int, uintptr_t>, Workspace> g_ws;

int get_workspace(size_t need, cudaStream_t stream, void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e);
    unsigned long long ctx = 0;
    e = attn::current_context_id(&ctx);
    if (e != cudaSuccess)
        return cuda_fail(e);
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    Workspace& w = g_ws[{dev, reinterpret_cast<uintptr_t>(stream)}];
    if (w.ptr && w.ctx != ctx)
        w = Workspace{};
    if (w.bytes < need) {
        if (w.ptr) {
            e = cudaFree(w.ptr);  // synchronous: earlier kernels using it have finished
            w.ptr = nullptr;
            w.bytes = 0;
            if (e != cudaSuccess)
                return cuda_fail(e);
        }
        const size_t grow = need + need / 4;
        e = cudaMalloc(&w.ptr, grow);
        if (e != cudaSuccess) {
            w.ptr = nullptr;
            return cuda_fail(e);
        }
        w.bytes = grow;
        w.ctx = ctx;
    }
    *out = w.ptr;
    return ATTN_OK;
}

int validate_decode(const void* q, const void* k_cache, const void* v_cache, void* out,
                    const int* block_tables, const int* seq_lens, int num_seqs, int H_q, int H_kv,
                    int D, int max_blocks_per_seq, int block_size)
{
    if (num_seqs < 0 || max_blocks_per_seq < 1 || check_heads(H_q, H_kv) != ATTN_OK)
        return ATTN_ERR_INVALID_ARG;
    if (D != attn::kHeadDim || block_size != attn::kPageSize)
        return ATTN_ERR_UNSUPPORTED;
    if (num_seqs == 0)
        return ATTN_OK;
    if (!q || !k_cache || !v_cache || !out || !block_tables || !seq_lens)
        return ATTN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return ATTN_ERR_INVALID_ARG;
    const size_t qbytes = (size_t)num_seqs * H_q * D * 2;
    if (overlap(out, qbytes, q, qbytes))
        return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

}  // namespace

int attn::record_cuda_error(cudaError_t e) { return cuda_fail(e); }

cudaError_t attn::current_context_id(unsigned long long* id)
{
    static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (!get_current || !get_id)
        return cudaErrorNotSupported;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS)
        return cudaErrorDeviceUninitialized;
    if (!ctx) {
        // the runtime makes its primary context current on a thread lazily;
        // selecting the current device again makes it current now
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess)
            e = cudaSetDevice(dev);
        if (e != cudaSuccess)
            return e;
        if (get_current(&ctx) != CUDA_SUCCESS || !ctx)
            return cudaErrorDeviceUninitialized;
    }
    if (get_id(ctx, id) != CUDA_SUCCESS)
        return cudaErrorDeviceUninitialized;
    return cudaSuccess;
}

namespace {
int prefill_checked(const void* Q, const void* K, const void* V, void* O, int B, int S, int H_q,
                    int H_kv, int D, int causal, int stall_tile, cudaStream_t stream)
{
    if (B < 0 || S < 0 || check_heads(H_q, H_kv) != ATTN_OK)
        return ATTN_ERR_INVALID_ARG;
    if (D != attn::kHeadDim)
        return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || S == 0)
        return ATTN_OK;
    if (!Q || !K || !V || !O)
        return ATTN_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16))
        return ATTN_ERR_INVALID_ARG;
    const size_t qbytes = (size_t)B * S * H_q * D * 2;
    const size_t kvbytes = (size_t)B * S * H_kv * D * 2;
    if (overlap(O, qbytes, Q, qbytes) || overlap(O, qbytes, K, kvbytes) ||
        overlap(O, qbytes, V, kvbytes))
        return ATTN_ERR_INVALID_ARG;
    const cudaError_t e = attn::launch_prefill(Q, K, V, O, B, S, H_q, H_kv, causal, stall_tile, stream);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}
int prefill_paged_checked(const void* Q, const void* k_cache, const void* v_cache, void* O,
                          const int* cu_seqlens_q, const int* seq_lens_kv, const int* block_tables,
                          int B, int max_seqlen_q, int total_q, int H_q, int H_kv, int D,
                          int max_blocks_per_seq, int block_size, long long num_blocks, int causal,
                          const attn::QueryPrologue* qp, cudaStream_t stream)
{
    if (B < 0 || max_seqlen_q < 0 || total_q < 0 || max_blocks_per_seq < 1 || num_blocks < 0 ||
        check_heads(H_q, H_kv) != ATTN_OK)
        return ATTN_ERR_INVALID_ARG;
    if (D != attn::kHeadDim || block_size != attn::kPageSize)
        return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || total_q == 0 || max_seqlen_q == 0)
        return ATTN_OK;
    if (num_blocks < 1 || !Q || !k_cache || !v_cache || !O || !cu_seqlens_q || !seq_lens_kv ||
        !block_tables)
        return ATTN_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(O, 16) ||
        !aligned(cu_seqlens_q, 4) || !aligned(seq_lens_kv, 4) || !aligned(block_tables, 4))
        return ATTN_ERR_INVALID_ARG;
    const size_t qbytes = (size_t)total_q * H_q * D * 2;
    const size_t cache_bytes = (size_t)num_blocks * H_kv * block_size * D * 2;
    if (overlap(O, qbytes, Q, qbytes) || overlap(O, qbytes, k_cache, cache_bytes) ||
        overlap(O, qbytes, v_cache, cache_bytes))
        return ATTN_ERR_INVALID_ARG;
    const cudaError_t e = attn::launch_prefill_paged(
        Q, k_cache, v_cache, O, cu_seqlens_q, seq_lens_kv, block_tables, B, max_seqlen_q, total_q,
        H_q, H_kv, max_blocks_per_seq, num_blocks, causal, qp, stream);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}
}  // namespace

extern "C" {

ATTN_API int attn_prefill(const void* Q, const void* K, const void* V, void* O, int B, int S,
                          int H_q, int H_kv, int D, int causal, cudaStream_t stream)
{
    return prefill_checked(Q, K, V, O, B, S, H_q, H_kv, D, causal, -1, stream);
}

ATTN_API int attn_prefill_paged(const void* Q, const void* k_cache, const void* v_cache, void* O,
                                const int* cu_seqlens_q, const int* seq_lens_kv,
                                const int* block_tables, int B, int max_seqlen_q, int total_q,
                                int H_q, int H_kv, int D, int max_blocks_per_seq, int block_size,
                                long long num_blocks, int causal, cudaStream_t stream)
{
    return prefill_paged_checked(Q, k_cache, v_cache, O, cu_seqlens_q, seq_lens_kv, block_tables, B,
                                 max_seqlen_q, total_q, H_q, H_kv, D, max_blocks_per_seq,
                                 block_size, num_blocks, causal, nullptr, stream);
}

ATTN_API int attn_prefill_paged_qk_norm_rope(const void* Q, const void* k_cache, const void* v_cache,
                                             void* O, const int* cu_seqlens_q,
                                             const int* seq_lens_kv, const int* block_tables,
                                             const void* q_weight, const float* cos_sin,
                                             int max_pos, float eps, int B, int max_seqlen_q,
                                             int total_q, int H_q, int H_kv, int D,
                                             int max_blocks_per_seq, int block_size,
                                             long long num_blocks, int causal, cudaStream_t stream)
{
    if (max_pos < 1 || !(eps >= 0.0f) || !std::isfinite(eps))
        return ATTN_ERR_INVALID_ARG;
    if (B > 0 && total_q > 0 && max_seqlen_q > 0) {
        if (!cos_sin || !aligned(cos_sin, 16) || !aligned(q_weight, 16))
            return ATTN_ERR_INVALID_ARG;
        const size_t qbytes = (size_t)total_q * H_q * D * 2;
        const size_t tbytes = (size_t)max_pos * D * sizeof(float);
        if (overlap(O, qbytes, cos_sin, tbytes) || (q_weight && overlap(O, qbytes, q_weight, (size_t)D * 2)))
            return ATTN_ERR_INVALID_ARG;
    }
    const attn::QueryPrologue qp{q_weight, cos_sin, max_pos, eps};
    return prefill_paged_checked(Q, k_cache, v_cache, O, cu_seqlens_q, seq_lens_kv, block_tables, B,
                                 max_seqlen_q, total_q, H_q, H_kv, D, max_blocks_per_seq,
                                 block_size, num_blocks, causal, &qp, stream);
}

ATTN_API int attn_debug_prefill_stall(const void* Q, const void* K, const void* V, void* O, int B,
                                      int S, int H_q, int H_kv, int D, int causal, int stall_tile,
                                      cudaStream_t stream)
{
    if (stall_tile < 0)
        return ATTN_ERR_INVALID_ARG;
    return prefill_checked(Q, K, V, O, B, S, H_q, H_kv, D, causal, stall_tile, stream);
}

ATTN_API size_t attn_decode_paged_workspace_bytes(int num_seqs, int H_q, int H_kv, int D,
                                                  int max_blocks_per_seq, int block_size,
                                                  int pages_per_split)
{
    if (num_seqs < 0 || max_blocks_per_seq < 1 || check_heads(H_q, H_kv) != ATTN_OK ||
        D != attn::kHeadDim || block_size != attn::kPageSize)
        return 0;
    return attn::decode_workspace_bytes(
        attn::make_decode_plan(num_seqs, H_q, H_kv, max_blocks_per_seq, pages_per_split));
}

ATTN_API int attn_decode_paged_ws(const void* q, const void* k_cache, const void* v_cache,
                                  void* out, const int* block_tables, const int* seq_lens,
                                  int num_seqs, int H_q, int H_kv, int D, int max_blocks_per_seq,
                                  int block_size, int pages_per_split, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream)
{
    const int v = validate_decode(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q,
                                  H_kv, D, max_blocks_per_seq, block_size);
    if (v != ATTN_OK || num_seqs == 0)
        return v;
    const attn::DecodePlan p =
        attn::make_decode_plan(num_seqs, H_q, H_kv, max_blocks_per_seq, pages_per_split);
    if (!workspace || !aligned(workspace, 256) ||
        workspace_bytes < attn::decode_workspace_bytes(p))
        return ATTN_ERR_WORKSPACE;
    const cudaError_t e = attn::launch_decode(p, q, k_cache, v_cache, out, block_tables, seq_lens,
                                              workspace, stream);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

ATTN_API int attn_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                               void* out, const int* block_tables, const int* seq_lens,
                               int num_seqs, int H_q, int H_kv, int D, int max_blocks_per_seq,
                               int block_size, cudaStream_t stream)
{
    const int v = validate_decode(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q,
                                  H_kv, D, max_blocks_per_seq, block_size);
    if (v != ATTN_OK || num_seqs == 0)
        return v;
    const attn::DecodePlan p = attn::make_decode_plan(num_seqs, H_q, H_kv, max_blocks_per_seq, 0);
    void* ws = nullptr;
    const size_t need = attn::decode_workspace_bytes(p);
    const int r = get_workspace(need, stream, &ws);
    if (r != ATTN_OK)
        return r;
    const cudaError_t e =
        attn::launch_decode(p, q, k_cache, v_cache, out, block_tables, seq_lens, ws, stream);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

ATTN_API int attn_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                            const long long* slot_mapping, int num_tokens, int H_kv, int D,
                            int block_size, long long num_blocks, cudaStream_t stream)
{
    if (num_tokens < 0 || H_kv < 1 || num_blocks < 0)
        return ATTN_ERR_INVALID_ARG;
    if (D != attn::kHeadDim || block_size != attn::kPageSize)
        return ATTN_ERR_UNSUPPORTED;
    if (num_tokens == 0)
        return ATTN_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping || !aligned(k_new, 16) ||
        !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8))
        return ATTN_ERR_INVALID_ARG;
    const size_t new_bytes = (size_t)num_tokens * H_kv * D * 2;
    const size_t cache_bytes = (size_t)num_blocks * H_kv * block_size * D * 2;
    if (overlap(k_cache, cache_bytes, k_new, new_bytes) || overlap(k_cache, cache_bytes, v_new, new_bytes) ||
        overlap(v_cache, cache_bytes, k_new, new_bytes) || overlap(v_cache, cache_bytes, v_new, new_bytes) ||
        overlap(k_cache, cache_bytes, v_cache, cache_bytes))
        return ATTN_ERR_INVALID_ARG;
    const cudaError_t e = attn::launch_kv_append(k_new, v_new, k_cache, v_cache, slot_mapping,
                                                 num_tokens, H_kv, num_blocks, stream);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

ATTN_API int attn_decode_paged_append(const void* q, const void* k_new, const void* v_new,
                                      void* k_cache, void* v_cache, void* out,
                                      const long long* slot_mapping, const int* block_tables,
                                      const int* seq_lens, int num_seqs, int H_q, int H_kv, int D,
                                      int max_blocks_per_seq, int block_size, long long num_blocks,
                                      cudaStream_t stream)
{
    const int v = validate_decode(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q,
                                  H_kv, D, max_blocks_per_seq, block_size);
    if (v != ATTN_OK || num_seqs == 0)
        return v;
    const int r = attn_kv_append(k_new, v_new, k_cache, v_cache, slot_mapping, num_seqs, H_kv, D,
                                 block_size, num_blocks, stream);
    if (r != ATTN_OK)
        return r;
    return attn_decode_paged(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q, H_kv,
                             D, max_blocks_per_seq, block_size, stream);
}

ATTN_API int attn_lse_combine(const float* O_part, const float* lse, void* out, int R,
                              int n_split, int D, cudaStream_t stream)
{
    if (R < 0 || n_split < 1)
        return ATTN_ERR_INVALID_ARG;
    if (D != attn::kHeadDim)
        return ATTN_ERR_UNSUPPORTED;
    if (R == 0)
        return ATTN_OK;
    if (!O_part || !lse || !out || !aligned(O_part, 16) || !aligned(lse, 4) || !aligned(out, 16))
        return ATTN_ERR_INVALID_ARG;
    const cudaError_t e = attn::launch_lse_combine(O_part, lse, out, R, n_split, stream);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

ATTN_API int attn_rope_cos_sin_table(float* cos_sin, int max_pos, int D, double base,
                                     cudaStream_t stream)
{
    if (max_pos < 0 || !(base > 0.0) || !std::isfinite(base))
        return ATTN_ERR_INVALID_ARG;
    if (D != attn::kHeadDim)
        return ATTN_ERR_UNSUPPORTED;
    if (max_pos == 0)
        return ATTN_OK;
    if (!cos_sin || !aligned(cos_sin, 16))
        return ATTN_ERR_INVALID_ARG;
    const cudaError_t e = attn::launch_rope_table(cos_sin, max_pos, base, stream);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

namespace {

// Checks shared by both prologue entry points.  Q may be null only where
// `q_optional` (the keys-only form of the append).
int validate_prologue(const void* Q, const void* K, const void* q_weight, const void* k_weight,
                      const float* cos_sin, int max_pos, const int* positions, int num_tokens,
                      int H_q, int H_kv, int D, float eps, bool q_optional = false)
{
    if (num_tokens < 0 || H_q < 1 || H_kv < 1 || max_pos < 1 || !(eps >= 0.0f) || !std::isfinite(eps))
        return ATTN_ERR_INVALID_ARG;
    if (D != attn::kHeadDim)
        return ATTN_ERR_UNSUPPORTED;
    if (num_tokens == 0)
        return ATTN_OK;
    if ((!Q && !q_optional) || !K || !cos_sin || !positions || !aligned(Q, 16) || !aligned(K, 16) ||
        !aligned(cos_sin, 16) || !aligned(positions, 4) || !aligned(q_weight, 16) ||
        !aligned(k_weight, 16))
        return ATTN_ERR_INVALID_ARG;
    const size_t qb = Q ? (size_t)num_tokens * H_q * D * 2 : 0, kb = (size_t)num_tokens * H_kv * D * 2;
    const size_t tb = (size_t)max_pos * D / 2 * sizeof(float) * 2, pb = (size_t)num_tokens * 4;
    const void* read_only[] = {q_weight, k_weight, cos_sin, positions};
    const size_t ro_bytes[] = {(size_t)D * 2, (size_t)D * 2, tb, pb};
    if (overlap(Q, qb, K, kb))
        return ATTN_ERR_INVALID_ARG;
    for (int i = 0; i < 4; i++)
        if (read_only[i] && (overlap(Q, qb, read_only[i], ro_bytes[i]) ||
                             overlap(K, kb, read_only[i], ro_bytes[i])))
            return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

}  // namespace

ATTN_API int attn_qk_norm_rope(void* Q, void* K, const void* q_weight, const void* k_weight,
                               const float* cos_sin, int max_pos, const int* positions,
                               int num_tokens, int H_q, int H_kv, int D, float eps,
                               cudaStream_t stream)
{
    const int v = validate_prologue(Q, K, q_weight, k_weight, cos_sin, max_pos, positions,
                                    num_tokens, H_q, H_kv, D, eps);
    if (v != ATTN_OK || num_tokens == 0)
        return v;
    if (H_q + H_kv > attn::kMaxPrologueRowsPerToken)
        return ATTN_ERR_UNSUPPORTED;
    const cudaError_t e = attn::launch_qk_norm_rope(Q, K, nullptr, K, q_weight, k_weight, cos_sin,
                                                    max_pos, positions, nullptr, nullptr, nullptr, 0,
                                                    num_tokens, H_q, H_kv, eps, stream);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

ATTN_API int attn_qk_norm_rope_append(void* Q, const void* K, const void* V, const void* q_weight,
                                      const void* k_weight, const float* cos_sin, int max_pos,
                                      const int* positions, const long long* slot_mapping,
                                      void* k_cache, void* v_cache, int num_tokens, int H_q,
                                      int H_kv, int D, int block_size, long long num_blocks,
                                      float eps, cudaStream_t stream)
{
    const int v = validate_prologue(Q, K, q_weight, k_weight, cos_sin, max_pos, positions,
                                    num_tokens, H_q, H_kv, D, eps, true);
    if (v != ATTN_OK)
        return v;
    if (block_size != attn::kPageSize || (Q ? H_q : 0) + 2 * H_kv > attn::kMaxPrologueRowsPerToken)
        return ATTN_ERR_UNSUPPORTED;
    if (num_blocks < 0)
        return ATTN_ERR_INVALID_ARG;
    if (num_tokens == 0)
        return ATTN_OK;
    if (!V || !slot_mapping || !k_cache || !v_cache || !aligned(V, 16) || !aligned(slot_mapping, 8) ||
        !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return ATTN_ERR_INVALID_ARG;
    const size_t qb = Q ? (size_t)num_tokens * H_q * D * 2 : 0, kb = (size_t)num_tokens * H_kv * D * 2;
    const size_t cb = (size_t)num_blocks * H_kv * block_size * D * 2;
    if (overlap(Q, qb, V, kb) || overlap(k_cache, cb, v_cache, cb))
        return ATTN_ERR_INVALID_ARG;
    const void* inputs[] = {Q, K, V, cos_sin, positions, slot_mapping, q_weight, k_weight};
    const size_t in_bytes[] = {qb, kb, kb, (size_t)max_pos * D * 4, (size_t)num_tokens * 4,
                               (size_t)num_tokens * 8, (size_t)D * 2, (size_t)D * 2};
    for (int i = 0; i < 8; i++)
        if (inputs[i] && (overlap(k_cache, cb, inputs[i], in_bytes[i]) ||
                          overlap(v_cache, cb, inputs[i], in_bytes[i])))
            return ATTN_ERR_INVALID_ARG;
    const cudaError_t e = attn::launch_qk_norm_rope(Q, K, V, nullptr, q_weight, k_weight, cos_sin,
                                                    max_pos, positions, slot_mapping, k_cache,
                                                    v_cache, num_blocks, num_tokens, H_q, H_kv,
                                                    eps, stream);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

ATTN_API int attn_release_workspace(void)
{
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    int prev = 0;
    cudaError_t first = cudaGetDevice(&prev);
    for (auto& kv : g_ws) {
        if (kv.second.ptr) {
            cudaError_t e = cudaSetDevice(kv.first.first);
            unsigned long long ctx = 0;
            if (e == cudaSuccess)
                e = attn::current_context_id(&ctx);
            // a buffer of a context that no longer exists went away with it
            if (e == cudaSuccess && ctx == kv.second.ctx)
                e = cudaFree(kv.second.ptr);
            if (e != cudaSuccess && first == cudaSuccess)
                first = e;
        }
    }
    g_ws.clear();
    cudaSetDevice(prev);
    return first == cudaSuccess ? ATTN_OK : cuda_fail(first);
}

ATTN_API int attn_get_device_error(int* code, int reset)
{
    if (!code)
        return ATTN_ERR_INVALID_ARG;
    int v = 0;
    const cudaError_t e = attn::read_device_error(&v, reset != 0);
    if (e != cudaSuccess)
        return cuda_fail(e);
    *code = v;
    if (v & attn::kDevErrTimeout)
        return ATTN_ERR_TIMEOUT;
    if (v)
        return ATTN_ERR_BAD_INPUT;
    return ATTN_OK;
}

ATTN_API int attn_last_cuda_error(void) { return t_last_cuda_error; }

ATTN_API const char* attn_status_string(int status)
{
    switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported size (head_dim must be 128, block_size 16)";
    case ATTN_ERR_CUDA: return "CUDA runtime error";
    case ATTN_ERR_TIMEOUT: return "a bounded device wait timed out";
    case ATTN_ERR_BAD_INPUT: return "bad block table or sequence length seen on the device";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
    }
}

ATTN_API int attn_version(void) { return 100; }

}  // extern "C"
