// decode.cu -- single-token attention over a paged KV cache: split-K main
// kernel + log-sum-exp combine kernel.
//
// Operation ("Tutorial: Adding a New Kernel to RL.cu", add-cuda-kernel page,
// include/kernels/attention.cuh, "Paged Attention -- Decode"): one query token
// per sequence attends to all seq_lens[n] keys of its context; key t of
// sequence n lives in physical block block_tables[n][t / 16], slot t % 16, of
// k_cache/v_cache [num_blocks, H_kv, 16, 128]; q head h reads kv head
// h*H_kv/H_q.  The split-K ("flash decoding") structure is the next step the
// "GRPO-CUDA Project Memory" page names under "Remaining Gap vs nano-vllm";
// the merge of partials by their log-sum-exp rests on the online-softmax
// identity worked through in the Kimi-K2.6 KernelBench trace.
//
// GB300 design.  The work is a stream of 4 KB page chunks per (page, kv head),
// read once, so it is HBM-bound while the arithmetic per byte stays low: 2
// FLOP per K/V byte for each query head that shares the kv head.
//  * One CTA (4 warps) per (sequence, kv head, chunk of up to 16 query heads,
//    split of `pages_per_split` pages).  Warps take pages round-robin.
//  * The query heads of a GQA group form the rows (zero-padded to 16) of a
//    warp-level tensor-core tile: per 16-key page a warp computes
//    S[16 x 16] = Q K^T with 16 m16n8k16 MMAs and O[16 x 128] += P V with 16
//    more, so every K/V byte is read from HBM once for all heads of its group
//    and the arithmetic stays a small fraction of a page's load time at any
//    group size (on CUDA cores it overtook the loads from four heads up).
//  * Pages reach shared memory by 16-byte asynchronous copies into a
//    two-stage ring per warp (3 CTAs and ~190 KB in flight per SM), rows
//    swizzled so the matrix loads that feed the MMAs are conflict-free.
//  * Scores are in log2 units (scale log2(e)/sqrt(D) applied to the FP32
//    scores); P is rounded to FP16 for the PV MMA; exp2 uses MUFU ex2.
//  * The CTA merges its 4 warps in shared memory and writes one partial
//    (O normalised, lse natural log) per head; the combine kernel merges the
//    splits.  A context that fits one split is finished by the main kernel
//    (FP16 output, no partial), and the combine leaves its rows alone.  Empty
//    splits (past the end of a sequence) exit at once and are skipped by the
//    combine, which recomputes the split count from seq_lens.
//  * The launches of a step (KV append, main kernel, combine) are chained by
//    programmatic dependent launch: each kernel lets its dependent be
//    scheduled as soon as its own CTAs have started, and the dependent waits on
//    the device for its results, so the launch gaps overlap the tails.
#include <cstdint>
#include <mutex>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "internal.h"
#include "ptx.cuh"

namespace attn {

__device__ int g_device_error = 0;

int* device_error_word()
{
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess)
        return nullptr;
    return static_cast<int*>(p);
}

cudaError_t read_device_error(int* out, bool reset)
{
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return e;
    e = cudaMemcpyFromSymbol(out, g_device_error, sizeof(int));
    if (e != cudaSuccess || !reset)
        return e;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

namespace {

constexpr int kDecodeWarps = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Programmatic dependent launch (sm_90+): a kernel launched with programmatic
// stream serialization may start before the previous kernel in the stream has
// finished; it must wait (grid_dependency_wait) before touching what that
// kernel writes.  A kernel lets its dependent start early with
// allow_dependents.  Both are no-ops without such a dependency.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void allow_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// The main kernel (the design notes at the top of the file).  Rows of the head
// tile past the group's heads are computed on zero queries and not written.
constexpr int kMmaHeads = 16;                       // tile rows: heads per CTA
constexpr int kMmaStages = 2;                       // pages in flight per warp
constexpr int kPageBytes = kPageSize * kHeadDim * 2;    // one (page, kv head) of K or V: 4 KB
constexpr int kMmaStageBytes = 2 * kPageBytes;          // K and V
constexpr int kMmaSmemBytes = kDecodeWarps * kMmaStages * kMmaStageBytes;   // 64 KB

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr) : "memory");
}
// D (16x8, FP32) += A (16x16, FP16, row) * B (16x8, FP16, col)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi)
{
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}
// byte offset of 16-byte chunk c of key row r in a swizzled 16 x 256-byte page
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 256 + ((c ^ (r & 7)) << 4)); }

__global__ void __launch_bounds__(kDecodeWarps * 32, 3)
decode_mma_kernel(const __half* __restrict__ q, const __half* __restrict__ k_cache,
                  const __half* __restrict__ v_cache, const int* __restrict__ block_tables,
                  const int* __restrict__ seq_lens, float* __restrict__ O_part,
                  float* __restrict__ lse_part, __half* __restrict__ out, int H_q, int H_kv,
                  int group, int chunks, int max_blocks_per_seq, int pages_per_split, int n_split,
                  float scale_log2)
{
    constexpr int D = kHeadDim;
    constexpr int BS = kPageSize;
    extern __shared__ __align__(128) unsigned char dsm[];
    grid_dependency_wait();   // the cache may have been written by the launch before (KV append)
    allow_dependents();       // the combine may be scheduled once every CTA has started
    const int split = blockIdx.x % n_split;
    int rest = blockIdx.x / n_split;
    const int chunk = rest % chunks;
    rest /= chunks;
    const int g = rest % H_kv;
    const int n = rest / H_kv;

    int L = seq_lens[n];
    const int max_len = max_blocks_per_seq * BS;
    if (L > max_len) {
        if (threadIdx.x == 0 && split == 0 && g == 0 && chunk == 0)
            atomicOr(&g_device_error, kDevErrSeqTooLong);
        L = max_len;
    }
    const int n_pages = (L + BS - 1) / BS;
    const int p_begin = split * pages_per_split;
    if (p_begin >= n_pages)
        return;  // empty split: the combine kernel does not read it
    const int p_end = min(n_pages, p_begin + pages_per_split);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int gid = lane >> 2;   // fragment row group
    const int tig = lane & 3;    // thread in group
    const int h0 = g * group + chunk * kMmaHeads;
    const int n_heads = min(kMmaHeads, group - chunk * kMmaHeads);

    // Q as A fragments, rows gid and gid + 8 (zero past the group), 8 K-steps of 16 dims
    uint32_t qa[8][4];
    {
        const bool v0 = gid < n_heads, v1 = gid + 8 < n_heads;
        // rows past the group read nothing (their pointers stay on row h0)
        const uint32_t* q0 = reinterpret_cast<const uint32_t*>(q + ((size_t)n * H_q + h0 + (v0 ? gid : 0)) * D);
        const uint32_t* q1 = reinterpret_cast<const uint32_t*>(q + ((size_t)n * H_q + h0 + (v1 ? gid + 8 : 0)) * D);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            qa[kk][0] = v0 ? q0[kk * 8 + tig] : 0u;
            qa[kk][1] = v1 ? q1[kk * 8 + tig] : 0u;
            qa[kk][2] = v0 ? q0[kk * 8 + 4 + tig] : 0u;
            qa[kk][3] = v1 ? q1[kk * 8 + 4 + tig] : 0u;
        }
    }

    const uint32_t ring = smem_u32(dsm) + warp * kMmaStages * kMmaStageBytes;
    const int* table = block_tables + (size_t)n * max_blocks_per_seq;
    const size_t page_stride = (size_t)H_kv * BS * D;  // halves per physical block

    // issue the copies of this warp's i-th page (an empty group for a bad or
    // missing one); V rows past the context are zeroed instead (their slots may
    // hold anything, and 0 * NaN would reach O through the MMA)
    auto issue = [&](int i) {
        const int p = p_begin + warp + i * kDecodeWarps;
        if (p < p_end) {
            const int phys = table[p];
            if (phys >= 0) {
                const int valid = min(BS, L - p * BS);
                const size_t base = (size_t)phys * page_stride + (size_t)g * BS * D;
                const uint32_t kst = ring + (i % kMmaStages) * kMmaStageBytes;
                const uint32_t vst = kst + kPageBytes;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int ci = lane + 32 * u;        // 16-byte chunk of the 4 KB page
                    const int r = ci >> 4, c = ci & 15;
                    cp_async16(kst + swz(r, c), k_cache + base + r * D + c * 8);
                    if (r < valid)
                        cp_async16(vst + swz(r, c), v_cache + base + r * D + c * 8);
                    else
                        asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(vst + swz(r, c)), "r"(0u) : "memory");
                }
            }
        }
        cp_async_commit();
    };

    float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F;   // rows gid, gid + 8 (log2 units)
    float l0 = 0.f, l1 = 0.f;                       // this thread's share of the row sums
    float o[16][4];
#pragma unroll
    for (int nb = 0; nb < 16; ++nb)
        o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;

    const int my_pages = p_begin + warp < p_end ? (p_end - p_begin - warp + kDecodeWarps - 1) / kDecodeWarps : 0;
#pragma unroll
    for (int i = 0; i < kMmaStages - 1; ++i)
        issue(i);
    for (int i = 0; i < my_pages; ++i) {
        issue(i + kMmaStages - 1);
        cp_async_wait<kMmaStages - 1>();
        __syncwarp();
        const int p = p_begin + warp + i * kDecodeWarps;
        const int phys = table[p];
        if (phys < 0) {
            if (lane == 0)
                atomicOr(&g_device_error, kDevErrBadBlockId);
            __syncwarp();
            continue;
        }
        const int valid = min(BS, L - p * BS);
        const uint32_t kst = ring + (i % kMmaStages) * kMmaStageBytes;
        const uint32_t vst = kst + kPageBytes;
        const int r8 = lane & 7, mi = lane >> 3;
        // S = Q K^T: n-blocks of keys 0-7 and 8-15
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t b0, b1, b2, b3;
            const int key = ((mi >> 1) << 3) + r8;
            ldsm_x4(kst + swz(key, (kk << 1) + (mi & 1)), b0, b1, b2, b3);
            mma16816(s[0], qa[kk], b0, b1);
            mma16816(s[1], qa[kk], b2, b3);
        }
        // online softmax over the page's keys (log2 units), rows gid and gid + 8
        float x[2][4];
#pragma unroll
        for (int nb = 0; nb < 2; ++nb)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = nb * 8 + tig * 2 + (e & 1);
                x[nb][e] = key < valid ? s[nb][e] * scale_log2 : -CUDART_INF_F;
            }
        float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
        float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);   // finite: key 0 of a page is valid
        const float a0 = ex2_approx(m0 - mn0), a1 = ex2_approx(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        float pr[2][4];
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
            pr[nb][0] = ex2_approx(x[nb][0] - mn0);
            pr[nb][1] = ex2_approx(x[nb][1] - mn0);
            pr[nb][2] = ex2_approx(x[nb][2] - mn1);
            pr[nb][3] = ex2_approx(x[nb][3] - mn1);
        }
        l0 = l0 * a0 + (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
        l1 = l1 * a1 + (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
        const uint32_t pa[4] = {pack_h2(pr[0][0], pr[0][1]), pack_h2(pr[0][2], pr[0][3]),
                                pack_h2(pr[1][0], pr[1][1]), pack_h2(pr[1][2], pr[1][3])};
        // O = O * alpha + P V, in n-blocks of 8 dims
#pragma unroll
        for (int nb = 0; nb < 16; nb += 2) {
            uint32_t b0, b1, b2, b3;
            const int key = ((mi & 1) << 3) + r8;
            ldsm_x4_t(vst + swz(key, nb + (mi >> 1)), b0, b1, b2, b3);
            o[nb][0] *= a0; o[nb][1] *= a0; o[nb][2] *= a1; o[nb][3] *= a1;
            o[nb + 1][0] *= a0; o[nb + 1][1] *= a0; o[nb + 1][2] *= a1; o[nb + 1][3] *= a1;
            mma16816(o[nb], pa, b0, b1);
            mma16816(o[nb + 1], pa, b2, b3);
        }
        __syncwarp();   // every lane has read this stage before it is refilled
    }
    cp_async_wait<0>();
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    __syncthreads();   // the rings are free: reuse them for the merge

    // merge the 4 warps through shared memory
    // rows padded to 136 floats: the 8-byte stores of a half-warp (4 rows x 4
    // pairs) then fall on distinct banks
    constexpr int SO = D + 8;
    float* sm_o = reinterpret_cast<float*>(dsm);                          // [warp][16][SO]
    float* sm_m = sm_o + kDecodeWarps * kMmaHeads * SO;                    // [warp][16]
    float* sm_l = sm_m + kDecodeWarps * kMmaHeads;                         // [warp][16]
#pragma unroll
    for (int nb = 0; nb < 16; ++nb) {
        const int d = nb * 8 + tig * 2;
        *reinterpret_cast<float2*>(&sm_o[(warp * kMmaHeads + gid) * SO + d]) = make_float2(o[nb][0], o[nb][1]);
        *reinterpret_cast<float2*>(&sm_o[(warp * kMmaHeads + gid + 8) * SO + d]) = make_float2(o[nb][2], o[nb][3]);
    }
    if (tig == 0) {
        sm_m[warp * kMmaHeads + gid] = m0;
        sm_m[warp * kMmaHeads + gid + 8] = m1;
        sm_l[warp * kMmaHeads + gid] = l0;
        sm_l[warp * kMmaHeads + gid + 8] = l1;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < n_heads * D; idx += blockDim.x) {
        const int hh = idx / D, d = idx % D;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w)
            M = fmaxf(M, sm_m[w * kMmaHeads + hh]);
        const size_t row = (size_t)n * H_q + h0 + hh;
        // a context of one split needs no combine: its output is final here
        const bool single = n_pages <= pages_per_split;
        if (M == -CUDART_INF_F) {
            // every page of this split had a negative block id: an empty segment
            if (single) {
                out[row * D + d] = __float2half_rn(0.f);
                continue;
            }
            O_part[(row * n_split + split) * D + d] = 0.f;
            if (d == 0)
                lse_part[row * n_split + split] = -CUDART_INF_F;
            continue;
        }
        float Lsum = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w) {
            const float c = ex2_approx(sm_m[w * kMmaHeads + hh] - M);  // 0 for a warp with no pages
            Lsum += c * sm_l[w * kMmaHeads + hh];
            acc += c * sm_o[(w * kMmaHeads + hh) * SO + d];
        }
        if (single) {
            out[row * D + d] = __float2half_rn(acc / Lsum);
            continue;
        }
        O_part[(row * n_split + split) * D + d] = acc / Lsum;
        if (d == 0)
            lse_part[row * n_split + split] = (M + __log2f(Lsum)) * kLn2;
    }
}

// One CTA of kCombineWarps warps per output row; lane owns 4 consecutive
// head-dim entries.  The warps take the row's splits round-robin (loads
// unrolled for memory-level parallelism) and are merged in shared memory.
// If seq_lens is given, row r = n*H_q + h uses the first
// ceil(ceil(seq_lens[n]/16)/pages_per_split) partials, and a row of one split
// is left alone (the main kernel wrote it); otherwise all n_split (partials
// with lse = -inf contribute nothing).
constexpr int kCombineWarps = 4;

__global__ void __launch_bounds__(kCombineWarps * 32)
lse_combine_kernel(const float* __restrict__ O_part, const float* __restrict__ lse_part,
                   __half* __restrict__ out, int n_split, const int* __restrict__ seq_lens,
                   int H_q, int pages_per_split, int max_len)
{
    constexpr int D = kHeadDim;
    constexpr int W = kCombineWarps;
    __shared__ float sm_max[W];
    __shared__ float sm_sum[W];
    __shared__ float4 sm_acc[W][32];
    grid_dependency_wait();   // the partials come from the launch before
    const int row = blockIdx.x;
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    int ns = n_split;
    if (seq_lens) {
        const int L = min(seq_lens[row / H_q], max_len);
        const int pages = (L + kPageSize - 1) / kPageSize;
        ns = (pages + pages_per_split - 1) / pages_per_split;
        if (ns == 1)
            return;   // the main kernel wrote this row's output itself
    }
    const float* lp = lse_part + (size_t)row * n_split;
    const float* op = O_part + (size_t)row * n_split * D + lane * 4;
    float M = -CUDART_INF_F;
    for (int i = threadIdx.x; i < ns; i += W * 32)
        M = fmaxf(M, lp[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (lane == 0)
        sm_max[warp] = M;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < W; ++k)
        M = fmaxf(M, sm_max[k]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (M != -CUDART_INF_F) {
        const float Ml = M * kLog2e;
        int i = warp;
        for (; i + 3 * W < ns; i += 4 * W) {
            float wt[4];
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                wt[u] = lp[i + u * W];
                v[u] = *reinterpret_cast<const float4*>(op + (size_t)(i + u * W) * D);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float w = ex2_approx(fmaf(wt[u], kLog2e, -Ml));
                wsum += w;
                acc.x = fmaf(w, v[u].x, acc.x);
                acc.y = fmaf(w, v[u].y, acc.y);
                acc.z = fmaf(w, v[u].z, acc.z);
                acc.w = fmaf(w, v[u].w, acc.w);
            }
        }
        for (; i < ns; i += W) {
            const float w = ex2_approx(fmaf(lp[i], kLog2e, -Ml));
            const float4 v = *reinterpret_cast<const float4*>(op + (size_t)i * D);
            wsum += w;
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
    }
    sm_acc[warp][lane] = acc;
    if (lane == 0)
        sm_sum[warp] = wsum;
    __syncthreads();
    if (warp == 0) {
        float tot = 0.f;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < W; ++k) {
            tot += sm_sum[k];
            a.x += sm_acc[k][lane].x;
            a.y += sm_acc[k][lane].y;
            a.z += sm_acc[k][lane].z;
            a.w += sm_acc[k][lane].w;
        }
        const float inv = tot > 0.f ? 1.f / tot : 0.f;  // all segments empty -> zeros
        __half2 h[2] = {__floats2half2_rn(a.x * inv, a.y * inv), __floats2half2_rn(a.z * inv, a.w * inv)};
        *reinterpret_cast<uint2*>(out + (size_t)row * D + lane * 4) = *reinterpret_cast<uint2*>(h);
    }
}

// The same merge with one warp per row, four rows per CTA: for rows of a few
// splits (the common case) the one-CTA-per-row form is dominated by launching
// and synchronising CTAs.  Each lane owns 4 head-dim entries.
__global__ void __launch_bounds__(kCombineWarps * 32)
lse_combine_rows_kernel(const float* __restrict__ O_part, const float* __restrict__ lse_part,
                        __half* __restrict__ out, int R, int n_split, const int* __restrict__ seq_lens,
                        int H_q, int pages_per_split, int max_len)
{
    constexpr int D = kHeadDim;
    grid_dependency_wait();   // the partials come from the launch before
    const int row = blockIdx.x * kCombineWarps + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (row >= R)
        return;
    int ns = n_split;
    if (seq_lens) {
        const int L = min(seq_lens[row / H_q], max_len);
        const int pages = (L + kPageSize - 1) / kPageSize;
        ns = (pages + pages_per_split - 1) / pages_per_split;
        if (ns == 1)
            return;   // the main kernel wrote this row's output itself
    }
    const float* lp = lse_part + (size_t)row * n_split;
    const float* op = O_part + (size_t)row * n_split * D + lane * 4;
    float M = -CUDART_INF_F;
    for (int i = lane; i < ns; i += 32)
        M = fmaxf(M, lp[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (M != -CUDART_INF_F) {
        const float Ml = M * kLog2e;
        int i = 0;
        for (; i + 3 < ns; i += 4) {
            float wt[4];
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                wt[u] = lp[i + u];
                v[u] = *reinterpret_cast<const float4*>(op + (size_t)(i + u) * D);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float w = ex2_approx(fmaf(wt[u], kLog2e, -Ml));
                wsum += w;
                acc.x = fmaf(w, v[u].x, acc.x);
                acc.y = fmaf(w, v[u].y, acc.y);
                acc.z = fmaf(w, v[u].z, acc.z);
                acc.w = fmaf(w, v[u].w, acc.w);
            }
        }
        for (; i < ns; ++i) {
            const float w = ex2_approx(fmaf(lp[i], kLog2e, -Ml));
            const float4 v = *reinterpret_cast<const float4*>(op + (size_t)i * D);
            wsum += w;
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;  // all segments empty -> zeros
    __half2 h[2] = {__floats2half2_rn(acc.x * inv, acc.y * inv), __floats2half2_rn(acc.z * inv, acc.w * inv)};
    *reinterpret_cast<uint2*>(out + (size_t)row * D + lane * 4) = *reinterpret_cast<uint2*>(h);
}

// Rows of at most this many splits are merged one warp per row.
constexpr int kRowsCombineMaxSplits = 8;

int pick_heads_per_cta(int) { return kMmaHeads; }

// SMs of the current device; a GB300's 152 if it cannot be queried (the
// workspace size may be asked for on a host without a GPU).
int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
        return n;
    cudaGetLastError();   // leave no error of the failed query for a later launch check
    return 152;
}

}  // namespace

DecodePlan make_decode_plan(int num_seqs, int H_q, int H_kv, int max_blocks_per_seq,
                            int pages_per_split)
{
    DecodePlan p{};
    p.num_seqs = num_seqs;
    p.H_q = H_q;
    p.H_kv = H_kv;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.group = H_q / H_kv;
    p.heads_per_cta = pick_heads_per_cta(p.group);
    p.chunks = (p.group + p.heads_per_cta - 1) / p.heads_per_cta;
    if (pages_per_split <= 0) {
        // 64 pages (1024 tokens) per split measured best (8 x 32k and H 64/8: +2 %
        // over 32; 256 mixed lengths level); smaller splits only when the grid
        // would otherwise hold fewer than 12 CTAs per SM of the current device
        // (4 waves of the 3 CTAs that fit on an SM).
        const long long kTargetCtas = 12LL * sm_count();
        const long long units = (long long)num_seqs * H_kv * p.chunks;
        pages_per_split = 64;
        while (pages_per_split > 4 &&
               units * ((max_blocks_per_seq + pages_per_split - 1) / pages_per_split) < kTargetCtas)
            pages_per_split /= 2;
    }
    p.pages_per_split = pages_per_split;
    p.n_split = (max_blocks_per_seq + pages_per_split - 1) / pages_per_split;
    const size_t rows = (size_t)num_seqs * H_q;
    p.o_part_bytes = rows * p.n_split * kHeadDim * sizeof(float);
    p.lse_part_bytes = rows * p.n_split * sizeof(float);
    return p;
}

size_t decode_workspace_bytes(const DecodePlan& p)
{
    const size_t a = (p.o_part_bytes + 255) & ~size_t(255);
    return a + ((p.lse_part_bytes + 255) & ~size_t(255));
}

// Launch configuration of a kernel that may start while the previous kernel in
// the stream finishes (it waits on the device before reading that kernel's output).
static void dependent_launch(cudaLaunchConfig_t& cfg, cudaLaunchAttribute (&attr)[1], dim3 grid, dim3 block,
                             cudaStream_t stream)
{
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
}

static cudaError_t launch_main_mma(const DecodePlan& p, const void* q, const void* k_cache,
                                   const void* v_cache, void* out, const int* block_tables,
                                   const int* seq_lens, float* O_part, float* lse_part, cudaStream_t stream)
{
    const long long grid = (long long)p.num_seqs * p.H_kv * p.chunks * p.n_split;
    if (grid > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    // the shared-memory opt-in is a per-context kernel attribute: set once per
    // device and context (a context that replaced one after a reset gets it too)
    static std::mutex mtx;
    static unsigned long long attr_ctx[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    unsigned long long ctx = 0;
    e = current_context_id(&ctx);
    if (e != cudaSuccess)
        return e;
    {
        std::lock_guard<std::mutex> lock(mtx);
        if (attr_ctx[dev] != ctx) {
            e = cudaFuncSetAttribute(decode_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMmaSmemBytes);
            if (e != cudaSuccess)
                return e;
            attr_ctx[dev] = ctx;
        }
    }
    const float scale_log2 = kLog2e / sqrtf((float)kHeadDim);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    dependent_launch(cfg, attr, dim3((unsigned)grid), dim3(kDecodeWarps * 32), stream);
    cfg.dynamicSmemBytes = kMmaSmemBytes;
    return cudaLaunchKernelEx(&cfg, decode_mma_kernel, static_cast<const __half*>(q),
                              static_cast<const __half*>(k_cache), static_cast<const __half*>(v_cache),
                              block_tables, seq_lens, O_part, lse_part, static_cast<__half*>(out), p.H_q,
                              p.H_kv, p.group, p.chunks, p.max_blocks_per_seq, p.pages_per_split, p.n_split,
                              scale_log2);
}

cudaError_t launch_decode(const DecodePlan& p, const void* q, const void* k_cache,
                          const void* v_cache, void* out, const int* block_tables,
                          const int* seq_lens, void* ws, cudaStream_t stream)
{
    float* O_part = static_cast<float*>(ws);
    float* lse_part = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                               ((p.o_part_bytes + 255) & ~size_t(255)));
    cudaError_t e = launch_main_mma(p, q, k_cache, v_cache, out, block_tables, seq_lens, O_part, lse_part, stream);
    if (e != cudaSuccess)
        return e;
    const int R = p.num_seqs * p.H_q;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    if (p.n_split <= kRowsCombineMaxSplits) {
        dependent_launch(cfg, attr, dim3((unsigned)((R + kCombineWarps - 1) / kCombineWarps)),
                         dim3(kCombineWarps * 32), stream);
        return cudaLaunchKernelEx(&cfg, lse_combine_rows_kernel, (const float*)O_part, (const float*)lse_part,
                                  static_cast<__half*>(out), R, p.n_split, seq_lens, p.H_q, p.pages_per_split,
                                  p.max_blocks_per_seq * kPageSize);
    }
    dependent_launch(cfg, attr, dim3((unsigned)R), dim3(kCombineWarps * 32), stream);
    return cudaLaunchKernelEx(&cfg, lse_combine_kernel, (const float*)O_part, (const float*)lse_part,
                              static_cast<__half*>(out), p.n_split, seq_lens, p.H_q, p.pages_per_split,
                              p.max_blocks_per_seq * kPageSize);
}

cudaError_t launch_lse_combine(const float* O_part, const float* lse_part, void* out, int R,
                               int n_split, cudaStream_t stream)
{
    if (n_split <= kRowsCombineMaxSplits)
        lse_combine_rows_kernel<<<(R + kCombineWarps - 1) / kCombineWarps, kCombineWarps * 32, 0, stream>>>(
            O_part, lse_part, static_cast<__half*>(out), R, n_split, nullptr, 1, 1, 0);
    else
        lse_combine_kernel<<<R, kCombineWarps * 32, 0, stream>>>(
            O_part, lse_part, static_cast<__half*>(out), n_split, nullptr, 1, 1, 0);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ KV append
//
// "GRPO-CUDA Project Memory" page, "KV Cache design": reshape-and-cache
// writes each new token's K/V row into its paged slot, slot_mapping[token] =
// physical_block * block_size + offset (int64), and skips slot -1 (padding
// tokens, "Known bugs fixed").  One CTA per token; 16-byte copies of the
// token's H_kv head rows of K and of V.  Slots outside [0, num_blocks*16)
// other than -1 are skipped and flagged.

__global__ void __launch_bounds__(128)
kv_append_kernel(const __half* __restrict__ k_new, const __half* __restrict__ v_new,
                 __half* __restrict__ k_cache, __half* __restrict__ v_cache,
                 const long long* __restrict__ slot_mapping, int H_kv, long long num_blocks)
{
    constexpr int D = kHeadDim;
    constexpr int BS = kPageSize;
    allow_dependents();
    const int t = blockIdx.x;
    const long long slot = slot_mapping[t];
    if (slot < 0 || slot >= num_blocks * BS) {
        if (slot != -1 && threadIdx.x == 0)
            atomicOr(&g_device_error, kDevErrBadSlot);
        return;
    }
    const long long block = slot / BS;
    const int pos = (int)(slot % BS);
    const int chunks = H_kv * D / 8;  // 16-byte chunks per row set
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
        const int g = c / (D / 8), d8 = c % (D / 8);
        const size_t src = ((size_t)t * H_kv + g) * D + d8 * 8;
        const size_t dst = (((size_t)block * H_kv + g) * BS + pos) * D + d8 * 8;
        *reinterpret_cast<uint4*>(k_cache + dst) = *reinterpret_cast<const uint4*>(k_new + src);
        *reinterpret_cast<uint4*>(v_cache + dst) = *reinterpret_cast<const uint4*>(v_new + src);
    }
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const long long* slot_mapping, int num_tokens, int H_kv,
                             long long num_blocks, cudaStream_t stream)
{
    kv_append_kernel<<<num_tokens, 128, 0, stream>>>(
        static_cast<const __half*>(k_new), static_cast<const __half*>(v_new),
        static_cast<__half*>(k_cache), static_cast<__half*>(v_cache), slot_mapping, H_kv, num_blocks);
    return cudaGetLastError();
}

}  // namespace attn
