// rope.cu -- the attention-input prologue: per-head QK-norm (RMSNorm) followed by
// the NeoX split-half rotary embedding, optionally fused with the KV append.
//
// What it computes ("GRPO-CUDA Project Memory" page, "Qwen3-Specific Notes" and
// "RoPE design"; angle definition from the Kimi-K2.6 KernelBench trace):
//   y[d]         = w[d] * x[d] / sqrt(mean(x^2) + eps)      (skipped when w is null)
//   out[i]       = y[i] c_i - y[i+64] s_i,   i < 64
//   out[i+64]    = y[i+64] c_i + y[i] s_i
//   (c_i, s_i)   = (cos, sin)(pos * base^(-2i/128)), read from an FP32 table
//
// The op streams q/k/v once (HBM-bound, no reuse), so the design is about bytes
// in flight and instructions per row, not tensor cores:
//  * each CTA owns a contiguous range of tokens; a producer warp copies them a
//    chunk at a time -- their contiguous q, k and v rows and the cos/sin rows of
//    their positions -- into a 4-stage shared-memory ring with bulk asynchronous
//    copies (cp.async.bulk, completion counted on an mbarrier per stage), so
//    ~150 KB per SM are in flight with no registers held;
//  * 16 consumer warps process rows out of shared memory, one row per 8-lane
//    group: lane m takes values 8m..8m+7 and their rotation partners 64+8m..,
//    so the rotation needs no shuffle and the sum of squares is a 3-step xor
//    reduction; results go straight to global memory (q in place, k and v to
//    their cache slots) with 16-byte stores;
//  * consumers release a stage with one arrive per warp; every wait is bounded.
//
// The rotation runs in FP32 on the table's FP32 (cos, sin); the table itself is
// built once in FP64 (pos * freq and sincos in double, then rounded), so the
// angle of a token at position 100k is as exact as that of position 1.  Table
// layout (per position, 32 float4 = 512 bytes, ordered so that the 8 lanes of a
// row read 128 contiguous bytes per load):
//   float4 index (p, i, m), i < 4, m < 8, at p*32 + i*8 + m holds
//   {cos a, cos b, sin a, sin b} of pairs a = 8m + 2i and b = a + 1.

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kD = kHeadDim;
constexpr int kRowBytes = kD * 2;                 // one FP16 row
constexpr int kTableRowBytes = kD / 2 * 8;        // 64 (cos, sin) FP32 pairs
constexpr int kConsumerWarps = 16;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kGroups = kConsumerWarps * 4;       // 8-lane row groups
constexpr int kStages = 4;
constexpr int kStageDataBudget = 48 * 1024;       // row + table bytes per stage
constexpr int kMaxChunk = 16;                     // tokens per stage
constexpr int kHeaderBytes = kMaxChunk * 12;      // positions + slots of the chunk

struct PrologueArgs {
    __half* q;                  // [T, H_q, 128], rewritten in place
    const __half* k;            // [T, H_kv, 128]
    const __half* v;            // [T, H_kv, 128]   (append only)
    __half* k_out;              // [T, H_kv, 128]   destination of k without append (== k)
    const __half* q_w;          // [128] or nullptr: no norm on q
    const __half* k_w;          // [128] or nullptr: no norm on k
    const float4* table;        // [max_pos, 32] float4, layout above
    const int* positions;       // [T]
    const long long* slots;     // [T] (append only)
    __half* k_cache;            // [num_blocks, H_kv, 16, 128] (append only)
    __half* v_cache;
    long long num_slots;        // num_blocks * 16
    int T, H_q, H_kv, max_pos;
    int R;                      // rows per token: H_q + H_kv (+ H_kv for v when appending)
    int chunk;                  // tokens per stage
    int n_chunks;
    int chunks_per_cta;         // each CTA takes a contiguous range of chunks
    float inv_R;                // 1/R, for the row -> (token, row-in-token) split
    int stage_bytes;            // one ring stage: rows, table rows, header
    float eps;
    int* err;
};

// Stage layout: [q rows chunk*H_q][k rows chunk*H_kv][v rows chunk*H_kv]
// [table rows chunk][header: int pos[kMaxChunk], long long slot[kMaxChunk]].
struct StageLayout {
    int k_off, v_off, table_off, pos_off, slot_off;
    __device__ explicit StageLayout(const PrologueArgs& a)
    {
        k_off = a.chunk * a.H_q * kRowBytes;
        v_off = k_off + a.chunk * a.H_kv * kRowBytes;
        table_off = a.chunk * a.R * kRowBytes;
        slot_off = table_off + a.chunk * kTableRowBytes;   // 256-byte aligned
        pos_off = slot_off + kMaxChunk * 8;
    }
};

__device__ __forceinline__ void h8_to_f(const uint4& u, float (&f)[8])
{
    const __half2* h = reinterpret_cast<const __half2*>(&u);
    #pragma unroll
    for (int c = 0; c < 4; c++) {
        const float2 p = __half22float2(h[c]);
        f[2 * c] = p.x;
        f[2 * c + 1] = p.y;
    }
}

__device__ __forceinline__ uint4 f_to_h8(const float (&f)[8])
{
    uint4 u;
    __half2* h = reinterpret_cast<__half2*>(&u);
    #pragma unroll
    for (int c = 0; c < 4; c++)
        h[c] = __floats2half2_rn(f[2 * c], f[2 * c + 1]);
    return u;
}

// Norm (when NORM) and rotation of one row held as lo = values 8m..8m+7 and
// hi = values 64+8m..64+8m+7 by lane m of an 8-lane group.
template <bool NORM>
__device__ __forceinline__ void rotate_row(float (&lo)[8], float (&hi)[8], const float (&wlo)[8],
                                           const float (&whi)[8], const float4 (&cs)[4],
                                           unsigned mask, float eps)
{
    if (NORM) {
        float ss = 0.f;
        #pragma unroll
        for (int e = 0; e < 8; e++) {
            ss = fmaf(lo[e], lo[e], ss);
            ss = fmaf(hi[e], hi[e], ss);
        }
        ss += __shfl_xor_sync(mask, ss, 4);
        ss += __shfl_xor_sync(mask, ss, 2);
        ss += __shfl_xor_sync(mask, ss, 1);
        const float inv = rsqrtf(ss * (1.0f / kD) + eps);
        #pragma unroll
        for (int e = 0; e < 8; e++) {
            lo[e] = (lo[e] * inv) * wlo[e];
            hi[e] = (hi[e] * inv) * whi[e];
        }
    }
    #pragma unroll
    for (int i = 0; i < 4; i++) {
        const float4 t = cs[i];   // {cos a, cos b, sin a, sin b}, pairs a = 8m+2i, b = a+1
        const float la = lo[2 * i], lb = lo[2 * i + 1], ha = hi[2 * i], hb = hi[2 * i + 1];
        lo[2 * i] = fmaf(la, t.x, -ha * t.z);
        lo[2 * i + 1] = fmaf(lb, t.y, -hb * t.w);
        hi[2 * i] = fmaf(ha, t.x, la * t.z);
        hi[2 * i + 1] = fmaf(hb, t.y, lb * t.w);
    }
}

// Add bytes to the transaction count of the current phase without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// The producer warp.  Each stage is filled in two steps: the chunk's q, k and v
// rows (which do not depend on positions) are issued one chunk ahead of its
// header and cos/sin rows, so the first copies leave at once and the position
// loads never stall the row stream.  The CTA's tokens are contiguous, so their
// positions and slots are read a 32-token window at a time, one token per lane,
// one window ahead of use; lane 0 picks each token's entry with a shuffle,
// writes the stage header and issues the copies.  The stage's single arrive
// comes last, after the header stores.
template <bool APPEND>
__device__ __forceinline__ void producer(const PrologueArgs& a, unsigned char* smem,
                                         uint64_t* full, uint64_t* empty, volatile int* abort,
                                         int lane)
{
    const StageLayout L(a);
    const int c_begin = blockIdx.x * a.chunks_per_cta;
    const int c_end = min(c_begin + a.chunks_per_cta, a.n_chunks);
    if (c_begin >= c_end)
        return;
    const int t_end = min(c_end * a.chunk, a.T);
    int win = c_begin * a.chunk;
    int cur_p = -1, nxt_p = -1;
    long long cur_s = -1, nxt_s = -1;
    if (win + lane < t_end) {
        cur_p = __ldg(a.positions + win + lane);
        if (APPEND)
            cur_s = __ldg(a.slots + win + lane);
    }
    if (win + 32 + lane < t_end) {
        nxt_p = __ldg(a.positions + win + 32 + lane);
        if (APPEND)
            nxt_s = __ldg(a.slots + win + 32 + lane);
    }

    // step 1 for chunk index i (0-based within the CTA's range): wait for its
    // stage to be free, then issue its q/k/v rows.  Lane 0 only; false on timeout.
    auto issue_rows = [&](int i) -> bool {
        const int s = i % kStages;
        if (i >= kStages && !mbar_wait(smem_u32(empty + s), ((i / kStages) - 1) & 1, abort))
            return false;
        const int t0 = (c_begin + i) * a.chunk;
        const int cn = min(a.chunk, a.T - t0);
        const uint32_t bar = smem_u32(full + s);
        const uint32_t dst = smem_u32(smem + s * a.stage_bytes);
        mbar_expect_tx(bar, (uint32_t)cn * a.R * kRowBytes);
        if (a.H_q)
            bulk_load(dst, a.q + (size_t)t0 * a.H_q * kD, (uint32_t)cn * a.H_q * kRowBytes, bar);
        bulk_load(dst + L.k_off, a.k + (size_t)t0 * a.H_kv * kD, (uint32_t)cn * a.H_kv * kRowBytes,
                  bar);
        if (APPEND)
            bulk_load(dst + L.v_off, a.v + (size_t)t0 * a.H_kv * kD,
                      (uint32_t)cn * a.H_kv * kRowBytes, bar);
        return true;
    };

    const int n = c_end - c_begin;
    int rows_issued = 0, done = 0;
    int ok = 1;
    if (lane == 0)
        ok = issue_rows(0);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    rows_issued = ok ? 1 : 0;
    for (int i = 0; ok && i < n; i++) {
        if (rows_issued < n) {
            int r = 1;
            if (lane == 0)
                r = issue_rows(rows_issued);
            if (!__shfl_sync(0xffffffffu, r, 0)) {
                ok = 0;
                break;
            }
            rows_issued++;
        }
        int stop = 0;
        if (lane == 0)
            stop = *abort;
        if (__shfl_sync(0xffffffffu, stop, 0)) {
            ok = 0;
            break;
        }
        // step 2 for chunk i: header, cos/sin rows, arrive
        const int s = i % kStages;
        unsigned char* st = smem + s * a.stage_bytes;
        int* hpos = reinterpret_cast<int*>(st + L.pos_off);
        long long* hslot = reinterpret_cast<long long*>(st + L.slot_off);
        const int t0 = (c_begin + i) * a.chunk;
        const int cn = min(a.chunk, a.T - t0);
        uint32_t table_bytes = 0;
        for (int c = 0; c < cn; c++) {
            int idx = t0 + c - win;
            if (idx >= 32) {     // next window; load the one after it
                win += 32;
                idx -= 32;
                cur_p = nxt_p;
                cur_s = nxt_s;
                if (win + 32 + lane < t_end) {
                    nxt_p = __ldg(a.positions + win + 32 + lane);
                    if (APPEND)
                        nxt_s = __ldg(a.slots + win + 32 + lane);
                }
            }
            const int p = __shfl_sync(0xffffffffu, cur_p, idx);
            const long long sl = APPEND ? __shfl_sync(0xffffffffu, cur_s, idx) : 0;
            if (lane == 0) {
                hpos[c] = p;
                if (APPEND)
                    hslot[c] = sl;
                if (p >= 0 && p < a.max_pos)
                    table_bytes += kTableRowBytes;
            }
        }
        if (lane == 0) {
            const uint32_t bar = smem_u32(full + s);
            const uint32_t dst = smem_u32(st);
            mbar_arrive_expect_tx(bar, table_bytes);   // the arrive releases the header stores
            // one copy per run of consecutive positions: a bulk copy has a fixed
            // cost of order a hundred cycles, too much to pay per 512-byte row
            for (int c = 0; c < cn;) {
                const int p = hpos[c];
                if (p < 0 || p >= a.max_pos) {
                    c++;
                    continue;
                }
                int e = c + 1;
                while (e < cn && hpos[e] == hpos[e - 1] + 1 && hpos[e] < a.max_pos)
                    e++;
                bulk_load(dst + L.table_off + c * kTableRowBytes, a.table + (size_t)p * 32,
                          (uint32_t)(e - c) * kTableRowBytes, bar);
                c = e;
            }
        }
        done = i + 1;
        __syncwarp();
    }
    if (lane == 0 && !ok) {
        // A wait ran out (or another role gave up): flag it, complete the arrival
        // of every stage whose rows are in flight without a header, and let all
        // copies already issued land before the CTA exits.
        atomicOr(a.err, kDevErrTimeout);
        *abort = 1;
        for (int i = done; i < rows_issued; i++)
            mbar_arrive(smem_u32(full + i % kStages));
        const int never = 0;
        for (int i = rows_issued > kStages ? rows_issued - kStages : 0; i < rows_issued; i++)
            mbar_wait(smem_u32(full + i % kStages), (i / kStages) & 1, &never);
    }
}

template <bool APPEND>
__global__ void __launch_bounds__(kThreads, 1) qk_norm_rope_kernel(const PrologueArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * a.stage_bytes);
    uint64_t* empty = full + kStages;
    volatile int* abort = reinterpret_cast<volatile int*>(empty + kStages);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(smem_u32(full + s), 1);
            mbar_init(smem_u32(empty + s), kConsumerWarps);
        }
        *abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        producer<APPEND>(a, smem, full, empty, abort, lane);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const StageLayout L(a);
    const int g = threadIdx.x >> 3;            // 8-lane row group
    const int m = threadIdx.x & 7;             // lane in the group
    const unsigned mask = 0xffu << (lane & 24);
    float wq_lo[8] = {}, wq_hi[8] = {}, wk_lo[8] = {}, wk_hi[8] = {};
    if (a.q_w) {
        h8_to_f(__ldg(reinterpret_cast<const uint4*>(a.q_w) + m), wq_lo);
        h8_to_f(__ldg(reinterpret_cast<const uint4*>(a.q_w) + 8 + m), wq_hi);
    }
    if (a.k_w) {
        h8_to_f(__ldg(reinterpret_cast<const uint4*>(a.k_w) + m), wk_lo);
        h8_to_f(__ldg(reinterpret_cast<const uint4*>(a.k_w) + 8 + m), wk_hi);
    }
    const int c_begin = blockIdx.x * a.chunks_per_cta;
    const int c_end = min(c_begin + a.chunks_per_cta, a.n_chunks);
    int used = 0;
    for (int chunk = c_begin; chunk < c_end; chunk++, used++) {
        const int s = used % kStages;
        if (!mbar_wait(smem_u32(full + s), (used / kStages) & 1, abort)) {
            if (!*abort)
                atomicOr(a.err, kDevErrTimeout);
            *abort = 1;
            return;
        }
        const unsigned char* st = smem + s * a.stage_bytes;
        const int* hpos = reinterpret_cast<const int*>(st + L.pos_off);
        const long long* hslot = reinterpret_cast<const long long*>(st + L.slot_off);
        const int t0 = chunk * a.chunk;
        const int cn = min(a.chunk, a.T - t0);
        const int n_rows = cn * a.R;
        __half* q_chunk = a.q + (size_t)t0 * a.H_q * kD;
        __half* k_chunk = APPEND ? nullptr : a.k_out + (size_t)t0 * a.H_kv * kD;
        for (int r = g; r < n_rows; r += kGroups) {
            // r < 16 * 192, so the float quotient is exact after truncation
            const int c = (int)(((float)r + 0.5f) * a.inv_R);
            const int k = r - c * a.R;
            const int p = hpos[c];
            if (p < 0 || p >= a.max_pos) {   // the whole token is skipped
                if (k == 0 && m == 0)
                    atomicOr(a.err, kDevErrBadPosition);
                continue;
            }
            const unsigned char* src;
            __half* dst;
            int kind;                        // 0 q, 1 k, 2 v
            if (k < a.H_q) {
                const int row = c * a.H_q + k;
                src = st + row * kRowBytes;
                dst = q_chunk + row * kD;
                kind = 0;
            } else {
                const bool is_v = APPEND && k >= a.H_q + a.H_kv;
                const int h = k - a.H_q - (is_v ? a.H_kv : 0);
                const int row = c * a.H_kv + h;
                src = st + (is_v ? L.v_off : L.k_off) + row * kRowBytes;
                kind = is_v ? 2 : 1;
                if (APPEND) {
                    const long long slot = hslot[c];
                    if (slot < 0 || slot >= a.num_slots) {
                        if (slot != -1 && k == a.H_q && m == 0)
                            atomicOr(a.err, kDevErrBadSlot);
                        continue;
                    }
                    const unsigned long long us = (unsigned long long)slot;
                    __half* cache = is_v ? a.v_cache : a.k_cache;
                    dst = cache + (((us / kPageSize) * a.H_kv + h) * kPageSize + us % kPageSize) * kD;
                } else {
                    dst = k_chunk + row * kD;
                }
            }
            const uint4 xlo = reinterpret_cast<const uint4*>(src)[m];
            const uint4 xhi = reinterpret_cast<const uint4*>(src)[8 + m];
            if (kind == 2) {                 // v: a plain copy into the cache
                reinterpret_cast<uint4*>(dst)[m] = xlo;
                reinterpret_cast<uint4*>(dst)[8 + m] = xhi;
                continue;
            }
            const float4* cs = reinterpret_cast<const float4*>(st + L.table_off + c * kTableRowBytes) + m;
            const float4 csr[4] = {cs[0], cs[8], cs[16], cs[24]};
            float lo[8], hi[8];
            h8_to_f(xlo, lo);
            h8_to_f(xhi, hi);
            if (kind == 0) {
                if (a.q_w)
                    rotate_row<true>(lo, hi, wq_lo, wq_hi, csr, mask, a.eps);
                else
                    rotate_row<false>(lo, hi, wq_lo, wq_hi, csr, mask, a.eps);
            } else {
                if (a.k_w)
                    rotate_row<true>(lo, hi, wk_lo, wk_hi, csr, mask, a.eps);
                else
                    rotate_row<false>(lo, hi, wk_lo, wk_hi, csr, mask, a.eps);
            }
            reinterpret_cast<uint4*>(dst)[m] = f_to_h8(lo);
            reinterpret_cast<uint4*>(dst)[8 + m] = f_to_h8(hi);
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(empty + s));
    }
}

__global__ void rope_table_kernel(float4* __restrict__ table, long long entries, double base)
{
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;   // (p, i, m)
    if (idx >= entries)
        return;
    const long long p = idx / 32;
    const int i = (int)(idx / 8 % 4), m = (int)(idx % 8);
    const int pa = 8 * m + 2 * i;
    double sa, ca, sb, cb;
    sincos((double)p * pow(base, -2.0 * pa / kD), &sa, &ca);
    sincos((double)p * pow(base, -2.0 * (pa + 1) / kD), &sb, &cb);
    table[idx] = make_float4((float)ca, (float)cb, (float)sa, (float)sb);
}

}  // namespace

cudaError_t launch_rope_table(float* cos_sin, int max_pos, double base, cudaStream_t stream)
{
    const long long entries = (long long)max_pos * 32;
    const int threads = 256;
    rope_table_kernel<<<(unsigned)((entries + threads - 1) / threads), threads, 0, stream>>>(
        reinterpret_cast<float4*>(cos_sin), entries, base);
    return cudaGetLastError();
}

cudaError_t launch_qk_norm_rope(void* q, const void* k, const void* v, void* k_out,
                                const void* q_w, const void* k_w, const float* cos_sin,
                                int max_pos, const int* positions, const long long* slot_mapping,
                                void* k_cache, void* v_cache, long long num_blocks, int T,
                                int H_q, int H_kv, float eps, cudaStream_t stream)
{
    PrologueArgs a;
    const bool append = k_cache != nullptr;
    if (!q)
        H_q = 0;   // keys (and values) only: the queries are normalised and rotated elsewhere
    a.q = static_cast<__half*>(q);
    a.k = static_cast<const __half*>(k);
    a.v = static_cast<const __half*>(v);
    a.k_out = static_cast<__half*>(k_out);
    a.q_w = static_cast<const __half*>(q_w);
    a.k_w = static_cast<const __half*>(k_w);
    a.table = reinterpret_cast<const float4*>(cos_sin);
    a.positions = positions;
    a.slots = slot_mapping;
    a.k_cache = static_cast<__half*>(k_cache);
    a.v_cache = static_cast<__half*>(v_cache);
    a.num_slots = num_blocks * kPageSize;
    a.T = T;
    a.H_q = H_q;
    a.H_kv = H_kv;
    a.max_pos = max_pos;
    a.R = H_q + H_kv * (append ? 2 : 1);
    if (a.R > kMaxPrologueRowsPerToken)
        return cudaErrorInvalidValue;
    const int per_token = a.R * kRowBytes + kTableRowBytes;
    a.chunk = kStageDataBudget / per_token;
    a.chunk = a.chunk < 1 ? 1 : (a.chunk > kMaxChunk ? kMaxChunk : a.chunk);
    a.n_chunks = (T + a.chunk - 1) / a.chunk;
    a.stage_bytes = (a.chunk * per_token + kHeaderBytes + 127) / 128 * 128;
    a.eps = eps;
    a.err = device_error_word();
    if (!a.err)
        return cudaErrorUnknown;
    const size_t smem = (size_t)kStages * a.stage_bytes + 2 * kStages * sizeof(uint64_t) + 16;

    int dev = 0, sms = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess)
        return e;
    if (smem > (size_t)optin || sms < 1)
        return cudaErrorInvalidValue;
    const void* fn = append ? reinterpret_cast<const void*>(qk_norm_rope_kernel<true>)
                            : reinterpret_cast<const void*>(qk_norm_rope_kernel<false>);
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    int per_sm = 0;
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, smem);
    if (e != cudaSuccess)
        return e;
    const int ctas = sms * (per_sm > 0 ? per_sm : 1);
    a.chunks_per_cta = (a.n_chunks + ctas - 1) / ctas;
    a.inv_R = 1.0f / (float)a.R;
    const int grid = (a.n_chunks + a.chunks_per_cta - 1) / a.chunks_per_cta;
    if (append)
        qk_norm_rope_kernel<true><<<grid, kThreads, smem, stream>>>(a);
    else
        qk_norm_rope_kernel<false><<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace attn
