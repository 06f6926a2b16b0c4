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
// read once: it is HBM-bound (~2 FLOP/byte), so the kernel is built for
// coalesced 16-byte loads and many bytes in flight, not for tensor cores.
//  * One CTA (4 warps) per (sequence, kv head, head chunk, split of
//    `pages_per_split` pages).  Warps take pages round-robin.
//  * All query heads of a GQA group that share the kv head are processed
//    against each loaded page, so every K/V byte is read from HBM once.
//  * Lane l of a warp owns tokens {l/16 + 2i} and head-dim slice
//    [(l%16)*8, +8) of a page: each load instruction of the warp covers two
//    full 256-byte token rows (coalesced), and every lane issues 8+8 16-byte
//    loads per page.
//  * Scores are in log2 units (q is pre-scaled by log2(e)/sqrt(D)); exp2 uses
//    the MUFU ex2 instruction.
//  * The CTA merges its 4 warps in shared memory and writes one partial
//    (O normalised, lse natural log) per head; the combine kernel merges the
//    splits.  Empty splits (past the end of a sequence) exit at once and are
//    skipped by the combine, which recomputes the split count from seq_lens.
//  * The launches of a step (KV append, main kernel, combine) are chained by
//    programmatic dependent launch: each kernel lets its dependent be
//    scheduled as soon as its own CTAs have started, and the dependent waits on
//    the device for its results, so the launch gaps overlap the tails.
#include <cstdint>
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

__device__ __forceinline__ uint4 ld_stream16(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8])
{
    const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __half22float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

// Sum over the 16 lanes of each half-warp.
__device__ __forceinline__ float half_warp_sum(float x)
{
    x += __shfl_xor_sync(0xffffffffu, x, 8);
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    return x;
}

// GP: query heads per CTA (>= 1).  Heads beyond the group are computed on
// zero queries and not written.
template <int GP>
__global__ void __launch_bounds__(kDecodeWarps * 32)
decode_splitk_kernel(const __half* __restrict__ q, const __half* __restrict__ k_cache,
                     const __half* __restrict__ v_cache, const int* __restrict__ block_tables,
                     const int* __restrict__ seq_lens, float* __restrict__ O_part,
                     float* __restrict__ lse_part, int H_q, int H_kv, int group, int chunks,
                     int max_blocks_per_seq, int pages_per_split, int n_split, float q_scale)
{
    constexpr int D = kHeadDim;
    constexpr int BS = kPageSize;
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
    const int half = lane / 16;         // token parity within a page
    const int dofs = (lane % 16) * 8;   // head-dim slice
    const int h0 = g * group + chunk * GP;
    const int n_heads = min(GP, group - chunk * GP);

    // this lane's query slices, pre-scaled so scores come out in log2 units
    float qf[GP][8];
#pragma unroll
    for (int hh = 0; hh < GP; ++hh) {
        if (hh < n_heads) {
            const uint4 v = *reinterpret_cast<const uint4*>(q + ((size_t)n * H_q + h0 + hh) * D + dofs);
            unpack8(v, qf[hh]);
#pragma unroll
            for (int d = 0; d < 8; ++d)
                qf[hh][d] *= q_scale;
        } else {
#pragma unroll
            for (int d = 0; d < 8; ++d)
                qf[hh][d] = 0.f;
        }
    }

    float m[GP], l[GP], o[GP][8];
#pragma unroll
    for (int hh = 0; hh < GP; ++hh) {
        m[hh] = -CUDART_INF_F;
        l[hh] = 0.f;
#pragma unroll
        for (int d = 0; d < 8; ++d)
            o[hh][d] = 0.f;
    }

    const int* table = block_tables + (size_t)n * max_blocks_per_seq;
    const size_t page_stride = (size_t)H_kv * BS * D;  // halves per physical block
    for (int p = p_begin + warp; p < p_end; p += kDecodeWarps) {
        int phys = table[p];
        const bool bad = phys < 0;
        if (bad) {
            if (lane == 0)
                atomicOr(&g_device_error, kDevErrBadBlockId);
            continue;
        }
        const size_t base = (size_t)phys * page_stride + (size_t)g * BS * D + dofs;
        const __half* kp = k_cache + base;
        const __half* vp = v_cache + base;
        uint4 kr[8], vr[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            kr[i] = ld_stream16(kp + (size_t)(half + 2 * i) * D);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            vr[i] = ld_stream16(vp + (size_t)(half + 2 * i) * D);

        const int valid = L - p * BS;  // tokens of this page inside the context (>= 1)
        // scores s[i][hh] for token half + 2i (identical on the 16 lanes of a half-warp)
        float s[8][GP];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float kf[8];
            unpack8(kr[i], kf);
#pragma unroll
            for (int hh = 0; hh < GP; ++hh) {
                float acc = 0.f;
#pragma unroll
                for (int d = 0; d < 8; ++d)
                    acc = fmaf(qf[hh][d], kf[d], acc);
                s[i][hh] = half_warp_sum(acc);
            }
        }
        // mask tokens past the end of the context (their slots may hold anything)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const bool in = (half + 2 * i) < valid;
#pragma unroll
            for (int hh = 0; hh < GP; ++hh)
                s[i][hh] = in ? s[i][hh] : -CUDART_INF_F;
            if (!in)
                vr[i] = make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int hh = 0; hh < GP; ++hh) {
            float mx = s[0][hh];
#pragma unroll
            for (int i = 1; i < 8; ++i)
                mx = fmaxf(mx, s[i][hh]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float m_new = fmaxf(m[hh], mx);   // finite: token 0 of a page is always valid
            const float alpha = ex2_approx(m[hh] - m_new);
            m[hh] = m_new;
            float psum = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                s[i][hh] = ex2_approx(s[i][hh] - m_new);
                psum += s[i][hh];
            }
            psum += __shfl_xor_sync(0xffffffffu, psum, 16);
            l[hh] = l[hh] * alpha + psum;
#pragma unroll
            for (int d = 0; d < 8; ++d)
                o[hh][d] *= alpha;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float vf[8];
            unpack8(vr[i], vf);
#pragma unroll
            for (int hh = 0; hh < GP; ++hh)
#pragma unroll
                for (int d = 0; d < 8; ++d)
                    o[hh][d] = fmaf(s[i][hh], vf[d], o[hh][d]);
        }
    }

    // lanes l and l^16 hold the same head-dim slice for the two token parities
#pragma unroll
    for (int hh = 0; hh < GP; ++hh)
#pragma unroll
        for (int d = 0; d < 8; ++d)
            o[hh][d] += __shfl_xor_sync(0xffffffffu, o[hh][d], 16);

    // merge the 4 warps through shared memory
    __shared__ float sm_o[kDecodeWarps][GP][D];
    __shared__ float sm_m[kDecodeWarps][GP], sm_l[kDecodeWarps][GP];
    if (lane < 16) {
#pragma unroll
        for (int hh = 0; hh < GP; ++hh)
#pragma unroll
            for (int d = 0; d < 8; ++d)
                sm_o[warp][hh][dofs + d] = o[hh][d];
    }
    if (lane == 0) {
#pragma unroll
        for (int hh = 0; hh < GP; ++hh) {
            sm_m[warp][hh] = m[hh];
            sm_l[warp][hh] = l[hh];
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < n_heads * D; idx += blockDim.x) {
        const int hh = idx / D, d = idx % D;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w)
            M = fmaxf(M, sm_m[w][hh]);
        const size_t row = (size_t)n * H_q + h0 + hh;
        if (M == -CUDART_INF_F) {
            // every page of this split had a negative block id (skipped and
            // flagged above): an empty segment, which the combine step weighs 0
            O_part[(row * n_split + split) * D + d] = 0.f;
            if (d == 0)
                lse_part[row * n_split + split] = -CUDART_INF_F;
            continue;
        }
        float Lsum = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w) {
            const float c = ex2_approx(sm_m[w][hh] - M);  // 0 for a warp with no pages
            Lsum += c * sm_l[w][hh];
            acc += c * sm_o[w][hh][d];
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
// ceil(ceil(seq_lens[n]/16)/pages_per_split) partials; otherwise all n_split
// (partials with lse = -inf contribute nothing).
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

int pick_heads_per_cta(int group)
{
    if (group <= 2)
        return group;
    if (group <= 4)
        return 4;
    return 8;
}

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
        // 32 pages (512 tokens) per split measured best on both decode
        // workloads; smaller splits only when the grid would otherwise hold
        // fewer than 16 CTAs per SM of the current device.
        const long long kTargetCtas = 16LL * sm_count();
        const long long units = (long long)num_seqs * H_kv * p.chunks;
        pages_per_split = 32;
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

template <int GP>
static cudaError_t launch_main(const DecodePlan& p, const void* q, const void* k_cache,
                               const void* v_cache, const int* block_tables, const int* seq_lens,
                               float* O_part, float* lse_part, cudaStream_t stream)
{
    const long long grid = (long long)p.num_seqs * p.H_kv * p.chunks * p.n_split;
    if (grid > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    const float q_scale = kLog2e / sqrtf((float)kHeadDim);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    dependent_launch(cfg, attr, dim3((unsigned)grid), dim3(kDecodeWarps * 32), stream);
    return cudaLaunchKernelEx(&cfg, decode_splitk_kernel<GP>, static_cast<const __half*>(q),
                              static_cast<const __half*>(k_cache), static_cast<const __half*>(v_cache),
                              block_tables, seq_lens, O_part, lse_part, p.H_q, p.H_kv, p.group, p.chunks,
                              p.max_blocks_per_seq, p.pages_per_split, p.n_split, q_scale);
}

cudaError_t launch_decode(const DecodePlan& p, const void* q, const void* k_cache,
                          const void* v_cache, void* out, const int* block_tables,
                          const int* seq_lens, void* ws, cudaStream_t stream)
{
    float* O_part = static_cast<float*>(ws);
    float* lse_part = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                               ((p.o_part_bytes + 255) & ~size_t(255)));
    cudaError_t e;
    switch (p.heads_per_cta) {
    case 1: e = launch_main<1>(p, q, k_cache, v_cache, block_tables, seq_lens, O_part, lse_part, stream); break;
    case 2: e = launch_main<2>(p, q, k_cache, v_cache, block_tables, seq_lens, O_part, lse_part, stream); break;
    case 4: e = launch_main<4>(p, q, k_cache, v_cache, block_tables, seq_lens, O_part, lse_part, stream); break;
    default: e = launch_main<8>(p, q, k_cache, v_cache, block_tables, seq_lens, O_part, lse_part, stream); break;
    }
    if (e != cudaSuccess)
        return e;
    const int R = p.num_seqs * p.H_q;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    dependent_launch(cfg, attr, dim3((unsigned)R), dim3(kCombineWarps * 32), stream);
    return cudaLaunchKernelEx(&cfg, lse_combine_kernel, (const float*)O_part, (const float*)lse_part,
                              static_cast<__half*>(out), p.n_split, seq_lens, p.H_q, p.pages_per_split,
                              p.max_blocks_per_seq * kPageSize);
}

cudaError_t launch_lse_combine(const float* O_part, const float* lse_part, void* out, int R,
                               int n_split, cudaStream_t stream)
{
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
