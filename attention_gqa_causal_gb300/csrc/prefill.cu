// prefill.cu -- causal / full grouped-query attention prefill on sm_103a
// tensor cores (tcgen05 + TMEM + TMA), over contiguous K/V or over a paged
// KV cache with packed variable-length query chunks.
//
// Operation ("Tutorial: Adding a New Kernel to RL.cu", add-cuda-kernel page,
// include/kernels/attention.cuh, "Flash Attention 2 -- Prefill"): Q,O are
// [B,S,H_q,D], K,V are [B,S,H_kv,D], FP16 in and out with FP32 accumulation;
// q head h reads kv head h*H_kv/H_q; with the causal mask token i attends to
// positions <= i; scale 1/sqrt(D).  The online-softmax recurrence (running
// max m, rescale factor exp(m_old - m_new), running sum l, final O/l) is the
// one the same page's kernel walks per key and the "GRPO-CUDA Project Memory"
// page summarises under "Attention kernel design"; here it runs per 128-key
// tile on tensor-core scores.
// The paged form takes K/V from the cache layout of the same header's "Paged
// Attention -- Decode" ([num_blocks, H_kv, 16, D] through block_tables) and
// packed query chunks whose first query sits after a cached prefix
// (L_kv - L_q keys): query i of a sequence attends to keys <= L_kv - L_q + i.
//
// GB300 design (one CTA per SM, 384 threads = three warpgroups):
//   warps 0-3  softmax of Q tile 0 (TMEM lanes 0..127 = its rows)
//   warps 4-7  softmax of Q tile 1
//   warp  8    MMA warp (one lane issues) + TMEM allocation
//   warp  9    TMA producer (one lane); it also initialises the barriers and
//              sends the first Q/K/V copies before the set-up barrier
//   warp 10    relay (one lane): adds "V_j and K_{j+1} landed" to tile 0's P
//              barrier, so the MMA warp checks one barrier per step
//   warp 11    idle (it completes the third warpgroup)
// After setup the warpgroups re-balance registers with setmaxnreg: the two
// softmax warpgroups rise to 200 per thread, the control warpgroup (MMA, TMA,
// relay) drops to 96.
// A CTA owns two 128-row Q tiles that read the same K/V: two query heads of
// one GQA group over the same rows when the group size is even (identical
// causal extents), else two consecutive row tiles of one head.  Per 128-key
// tile j the MMA warp computes S_t = Q_t K_j^T into TMEM (FP32), the softmax
// warps of tile t turn S_t into P_t = exp2(S*c - m) and write P_t back over
// S_t in TMEM as FP16, and the MMA warp accumulates O_t += P_t V_j with A read
// from TMEM.  The two tiles ping-pong: while one tile runs its softmax the
// tensor core works on the other.
// The row maximum is kept lazily: m is a reference that only moves when the
// row max exceeds it by more than kRescaleThreshold (log2 units); O and l
// always refer to the same m, so the result is exact.  Because m rarely moves
// after the first key tile, the exponentials of a tile are computed
// optimistically against the current m, and in the common case the tile's max
// is not reduced at all: every p of a row is at most the row's sum, so a sum
// within 2^kRescaleThreshold proves that no p went past the threshold.  Only
// when a row's sum exceeds it does the warp reload S (still intact in TMEM: P
// has not been written yet), take the tile max, move m if it grew past the
// threshold (rescaling O) and recompute.  This keeps the max reduction off the
// path from "S ready" to "P ready" that the tensor core waits for.
// TMEM: S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512) columns.
// SMEM: Q0,Q1 (32 KB each), 2 K stages, 2 V stages (32 KB each), all
// 128-byte swizzled as written by TMA boxes of 64 x 128 (contiguous K/V) or
// 64 x 16 (one cache page).  At the end O_t goes, normalised and swizzled,
// into Q_t's buffer (free once the last S GEMM has completed) and out by TMA
// store.  Key tiles wholly above the diagonal are never loaded or multiplied;
// only the diagonal tile is masked.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per tile
constexpr int D = kHeadDim;
constexpr int kPagesPerTile = BN / kPageSize;
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
constexpr int kRelayWarp = 10;   // folds the step's operand waits into tile 0's P barrier
constexpr int kThreads = 12 * 32;   // warp 11 only completes the third warpgroup
// Registers per thread after the warpgroups re-balance (setmaxnreg): the MMA/TMA
// warpgroup gives up what the softmax needs to keep a whole 128-key row of S
// in flight (at 168 registers its exp loop serialises).  Launch pool: 384
// threads x 168 = 64512 >= 256 x kSoftmaxRegs + 128 x kControlRegs = 63488,
// and per SM sub-partition (3 warps) 200 + 200 + 96 <= 512.  The host checks
// the compiled register count before launching (an increase that the pool
// cannot cover would wait forever).
constexpr int kSoftmaxRegs = 200;
constexpr int kControlRegs = 96;
static_assert(256 * kSoftmaxRegs + 128 * kControlRegs <= kThreads * 168, "register re-balance exceeds the launch pool");
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr uint32_t kTileBytes = BM * D * 2;      // 32 KB
constexpr uint32_t kBoxBytes = kTileBytes / 2;   // 16 KB: 128 rows x 64 halves
constexpr uint32_t kPageBoxBytes = kPageSize * 64 * 2;  // 2 KB: 16 rows x 64 halves
constexpr uint32_t kSmemQ = 0;
constexpr uint32_t kSmemK = 2 * kTileBytes;
constexpr uint32_t kSmemV = kSmemK + kKStages * kTileBytes;
constexpr uint32_t kSmemBytes = kSmemV + kVStages * kTileBytes;
constexpr uint32_t kSmemMax = 232448;               // 227 KB: the per-CTA opt-in limit
constexpr float kRescaleThreshold = 8.0f;
constexpr float kSumLimit = 256.0f;   // 2^kRescaleThreshold
constexpr float kLog2e = 1.4426950408889634f;

struct PrefillArgs {
    __half* O;
    int* err;
    int B, S, H_q, H_kv;   // B: batch (contiguous) or number of sequences (paged); S unused when paged
    int group;          // H_q / H_kv
    int head_pairs;     // 1: the two tiles are two heads; 0: two row tiles of one head
    int units_per_mb;   // B * H_kv * (tile pairs per kv head)
    int n_mb;           // number of row blocks (of the longest chunk when paged)
    int groups_per_super;  // (batch, kv head) groups per super-group of the causal / paged order
    int causal;
    float scale_log2;   // log2(e) / sqrt(D)
    int stall_tile;     // failure-detection test only: key tile whose K load is withheld (-1: none)
    // paged form only
    const int* cu_q;          // [B+1] query chunk offsets into packed Q / O
    const int* seq_lens_kv;   // [B] context lengths (prefix + chunk)
    const int* block_tables;  // [B, max_blocks]
    int max_blocks;
    int total_q;              // rows of packed Q / O
    // paged form with the query prologue folded in (rope != 0): each Q row is
    // normalised (q_w, nullptr = no norm) and rotated at its position in shared
    // memory before the first score GEMM
    int rope;
    const __half* q_w;        // [128] RMSNorm weight or nullptr
    const float4* rope_table; // [max_pos, 32] float4, the cos/sin table of attn_rope_cos_sin_table
    int max_pos;
    float eps;
};

struct Unit {
    int b, g, head[2], row0[2], n_kv;
    int q_base;  // first packed row of the sequence (paged) or b*S (contiguous)
    int Lq, Lkv, off;  // chunk length, context length, off = Lkv - Lq (position of query 0)
    int n_pages;
    int flags;   // device error bits found while decoding the unit
    bool valid;
};

template <bool PAGED>
__device__ __forceinline__ Unit decode_unit(const PrefillArgs& a, int u)
{
    Unit w;
    int mb, r;
    if (!PAGED && !a.causal) {
        // full attention, all units alike: (batch, kv head, pair) major, row
        // blocks minor, so the CTAs that read the same K/V run together and
        // fetch it from DRAM fewer times
        r = u / a.n_mb;
        mb = u % a.n_mb;
    } else {
        // causal (and paged): the (batch, kv head) groups are taken a super-group
        // at a time, so that the K/V the running CTAs read stays in L2 until
        // every row block of its group has passed over it; inside a
        // super-group longest row blocks come first, so short ones fill the
        // tail of the grid
        const int per_g = a.units_per_mb / (a.B * a.H_kv);
        const int n_groups = a.B * a.H_kv;
        const int units_per_super = a.n_mb * a.groups_per_super * per_g;
        const int sup = u / units_per_super;
        const int v = u - sup * units_per_super;
        const int per_mb_here = min(a.groups_per_super, n_groups - sup * a.groups_per_super) * per_g;
        mb = a.causal ? a.n_mb - 1 - v / per_mb_here : v / per_mb_here;
        r = sup * a.groups_per_super * per_g + v % per_mb_here;
    }
    const int per_g = a.units_per_mb / (a.B * a.H_kv);
    const int pr = r % per_g;
    r /= per_g;
    w.g = r % a.H_kv;
    w.b = r / a.H_kv;
    if (a.head_pairs) {
        w.head[0] = w.g * a.group + 2 * pr;
        w.head[1] = w.head[0] + 1;
        w.row0[0] = w.row0[1] = mb * BM;
    } else {
        w.head[0] = w.head[1] = w.g * a.group + pr;
        w.row0[0] = mb * 2 * BM;
        w.row0[1] = w.row0[0] + BM;
    }
    w.flags = 0;
    w.valid = true;
    if (!PAGED) {
        w.q_base = w.b * a.S;
        w.Lq = w.Lkv = a.S;
    } else {
        const int c0 = a.cu_q[w.b], c1 = a.cu_q[w.b + 1];
        // a chunk whose rows are not inside packed Q / O is flagged and becomes
        // empty (skipped below)
        const bool rows_ok = c0 >= 0 && c1 >= c0 && c1 <= a.total_q;
        w.q_base = rows_ok ? c0 : 0;
        w.Lq = rows_ok ? c1 - c0 : 0;
        if (!rows_ok)
            w.flags |= kDevErrBadLengths;
        w.Lkv = a.seq_lens_kv[w.b];
        const int max_len = a.max_blocks * kPageSize;
        if (w.Lkv > max_len) {
            w.flags |= kDevErrSeqTooLong;
            w.Lkv = max_len;
        }
        if (w.Lq < 0 || w.Lq > w.Lkv) {
            w.flags |= kDevErrBadLengths;
            w.valid = false;
        }
        if (w.Lq > a.n_mb * (a.head_pairs ? BM : 2 * BM))
            w.flags |= kDevErrBadLengths;  // longer than max_seqlen_q: its tail rows are not computed
        if (w.row0[0] >= w.Lq)
            w.valid = false;  // this row block is past the end of the chunk
    }
    w.off = w.Lkv - w.Lq;
    w.n_pages = (w.Lkv + kPageSize - 1) / kPageSize;
    const int last_row = min(w.Lq - 1, w.row0[1] + BM - 1);
    const int all_tiles = (w.Lkv + BN - 1) / BN;
    w.n_kv = a.causal ? min((w.off + last_row) / BN + 1, all_tiles) : all_tiles;
    return w;
}

struct SmemCtl {
    uint64_t q_full;
    uint64_t q0_full;        // Q tile 0 landed (without the query prologue; q_full then covers tile 1)
    uint64_t q_ready[2];     // tile t's rows normalised and rotated (query prologue folded in; 128 arrivals)
    uint64_t k_full[kKStages], k_empty[kKStages];
    uint64_t v_full[kVStages], v_empty[kVStages];
    uint64_t s_full[2], p_full[2], o_full[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
};

// Dynamic shared memory: the 1024-aligned tiles, then the control block.  The
// whole 227 KB is requested; the alignment padding the layout can absorb is
// what is left over (the kernel checks it at run time).
// After it, the query prologue's RMSNorm weight row (256 bytes, bulk-copied
// with the Q tiles).
constexpr uint32_t kSmemAlloc = kSmemMax;
constexpr uint32_t kSmemW = (kSmemBytes + (uint32_t)sizeof(SmemCtl) + 127u) & ~127u;
constexpr uint32_t kSmemEnd = kSmemW + D * 2;
constexpr uint32_t kAlignSlack = kSmemMax - kSmemEnd;
static_assert(kSmemEnd <= kSmemMax, "shared memory layout too large");

template <int N>
__device__ __forceinline__ void regs_increase()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

template <int N>
__device__ __forceinline__ void regs_decrease()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void flag_abort(SmemCtl* c, int* err)
{
    c->abort = 1;
    atomicOr(err, kDevErrTimeout);
}

// Max over 32 values: independent chains of 3-input max, then a small tree.
__device__ __forceinline__ float max32(const uint32_t (&r)[32])
{
    float m[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int b = k * 8;
        m[k] = fmax3(fmax3(__uint_as_float(r[b]), __uint_as_float(r[b + 1]), __uint_as_float(r[b + 2])),
                     fmax3(__uint_as_float(r[b + 3]), __uint_as_float(r[b + 4]), __uint_as_float(r[b + 5])),
                     fmaxf(__uint_as_float(r[b + 6]), __uint_as_float(r[b + 7])));
    }
    return fmaxf(fmax3(m[0], m[1], m[2]), m[3]);
}

// Per-head QK-norm then NeoX RoPE of Q rows, in place in the Q tiles, by the
// softmax warpgroups.  The arithmetic is the prologue's ("GRPO-CUDA Project
// Memory" page, "Qwen3-Specific Notes" and "RoPE design"): y = w x /
// sqrt(mean(x^2) + eps) in FP32 (no norm when w is null), then
// out_i = y_i c - y_{i+64} s, out_{i+64} = y_{i+64} c + y_i s with (c, s) of
// pair i at the row's position, rounded once to FP16.
// Work split: 8 lanes per row, 4 rows per warp at a time.  Lane m of a group
// owns the row's chunk m of both halves (elements 8m.. and their partners
// 64+8m..), which in a tile's 128-byte-swizzled boxes sit at ((m ^ row % 8) <<
// 4) of box 0 and box 1: no lane needs another's values except for the sum of
// squares (a 3-step xor reduction).  The lane's cos/sin entries of a row are
// entries i*8 + m (i < 4) of the table row, so a group reads 128 contiguous
// bytes per load.  When the two tiles are two heads over the same rows, a row
// index has one position in both, so each table row is fetched once: warpgroup
// t takes rows [64t, 64t + 64) of both tiles (4 passes); otherwise warpgroup t
// takes all 128 rows of its own tile (8 passes).
// Mixed-precision FMA (sm_100+): d = a * b + c with FP16 a, b and FP32 c, d;
// the product of two halves is exact in FP32, so no conversion is needed.
__device__ __forceinline__ float fma_hhf(uint16_t a, uint16_t b, float c)
{
    float d;
    asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
    return d;
}

// FP16 -> FP32 (exact) as an addition of +0 on the FMA path.
__device__ __forceinline__ float h2f(uint16_t a)
{
    float d;
    asm("add.rn.f32.f16 %0, %1, %2;" : "=f"(d) : "h"(a), "f"(0.f));
    return d;
}

__device__ __forceinline__ uint16_t half_bits(const uint4& u, int e)
{
    const uint32_t w = e < 2 ? u.x : e < 4 ? u.y : e < 6 ? u.z : u.w;
    return static_cast<uint16_t>((e & 1) ? w >> 16 : w & 0xffffu);
}

// One batch of N rows of this lane (row n of tile tile[n], table entries of
// pass pass[n]): all loads first, then the sums of squares and their group
// reductions interleaved over the rows, then the rotations and the stores (bit
// n of `store`), so that the rows' latencies overlap.  The halves enter the
// FP32 arithmetic through mixed-precision FMAs (x*x for the sum of squares,
// x*w, exact, before the 1/rms factor), which avoids the narrow FP16->FP32
// conversion path; each output is rounded once to FP16.
template <int N, int P>
__device__ __forceinline__ void norm_rope_batch(uint8_t* q_tiles, const int (&row)[N], const int (&tile)[N],
                                                const int (&pass)[N], const float4 (&cs)[P][4],
                                                uint32_t store, const uint4& w_lo, const uint4& w_hi,
                                                bool norm, float eps, int lane)
{
    const int m = lane % 8;
    const unsigned mask = 0xffu << (lane & 24);
    uint32_t off_lo[N];
    uint4 xl[N], xh[N];
#pragma unroll
    for (int n = 0; n < N; ++n) {
        off_lo[n] = tile[n] * kTileBytes + row[n] * 128 + ((m ^ (row[n] % 8)) << 4);
        xl[n] = *reinterpret_cast<const uint4*>(q_tiles + off_lo[n]);
        xh[n] = *reinterpret_cast<const uint4*>(q_tiles + off_lo[n] + kBoxBytes);
    }
    float ss[N];
    if (norm) {
#pragma unroll
        for (int n = 0; n < N; ++n) {
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;   // short independent chains
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                s0 = fma_hhf(half_bits(xl[n], e), half_bits(xl[n], e), s0);
                s1 = fma_hhf(half_bits(xl[n], e + 1), half_bits(xl[n], e + 1), s1);
                s2 = fma_hhf(half_bits(xh[n], e), half_bits(xh[n], e), s2);
                s3 = fma_hhf(half_bits(xh[n], e + 1), half_bits(xh[n], e + 1), s3);
            }
            ss[n] = (s0 + s1) + (s2 + s3);
        }
#pragma unroll
        for (int o = 4; o > 0; o >>= 1)
#pragma unroll
            for (int n = 0; n < N; ++n)
                ss[n] += __shfl_xor_sync(mask, ss[n], o);
    }
#pragma unroll
    for (int n = 0; n < N; ++n) {
        float lo[8], hi[8];
        if (norm) {
            const float inv = rsqrtf(ss[n] * (1.0f / D) + eps);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                lo[e] = fma_hhf(half_bits(xl[n], e), half_bits(w_lo, e), 0.f) * inv;
                hi[e] = fma_hhf(half_bits(xh[n], e), half_bits(w_hi, e), 0.f) * inv;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                lo[e] = h2f(half_bits(xl[n], e));
                hi[e] = h2f(half_bits(xh[n], e));
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 t = cs[pass[n]][i];   // {cos a, cos b, sin a, sin b}, pairs a = 8m + 2i, b = a + 1
            const float la = lo[2 * i], lb = lo[2 * i + 1], ha = hi[2 * i], hb = hi[2 * i + 1];
            lo[2 * i] = fmaf(la, t.x, -ha * t.z);
            lo[2 * i + 1] = fmaf(lb, t.y, -hb * t.w);
            hi[2 * i] = fmaf(ha, t.x, la * t.z);
            hi[2 * i + 1] = fmaf(hb, t.y, lb * t.w);
        }
        if (store >> n & 1u) {
            uint4 olo, ohi;
            olo.x = pack_half2(lo[0], lo[1]); olo.y = pack_half2(lo[2], lo[3]);
            olo.z = pack_half2(lo[4], lo[5]); olo.w = pack_half2(lo[6], lo[7]);
            ohi.x = pack_half2(hi[0], hi[1]); ohi.y = pack_half2(hi[2], hi[3]);
            ohi.z = pack_half2(hi[4], hi[5]); ohi.w = pack_half2(hi[6], hi[7]);
            *reinterpret_cast<uint4*>(q_tiles + off_lo[n]) = olo;
            *reinterpret_cast<uint4*>(q_tiles + off_lo[n] + kBoxBytes) = ohi;
        }
    }
}

// Row of pass p for this lane: shared rows (both tiles, warpgroup t's half) or
// the own tile's 128 rows.
__device__ __forceinline__ int rope_row(bool shared, int t, int p, int quad, int lane)
{
    return (shared ? 64 * t : 0) + p * 16 + quad * 4 + lane / 8;
}

// P = exp2(S*c - m) for 32 columns, packed in place (column pair -> even slot);
// adds the FP32 values into the 4 packed partial sums rs.
__device__ __forceinline__ void exp_pack32(uint32_t (&r)[32], float c, float neg_m, float (&rs)[8])
{
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        float x0, x1;
        ffma2(x0, x1, __uint_as_float(r[i]), __uint_as_float(r[i + 1]), c, c, neg_m, neg_m);
        const float p0 = ex2_approx(x0);
        const float p1 = ex2_approx(x1);
        const int k = (i / 2) % 4;
        fadd2(rs[2 * k], rs[2 * k + 1], p0, p1);
        r[i] = pack_half2(p0, p1);
    }
}

template <bool PAGED>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
               const PrefillArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    if (sbase - raw > kAlignSlack) {
        // the aligned layout would not fit: do nothing rather than overrun
        if (threadIdx.x == 0)
            atomicOr(a.err, kDevErrSmemLayout);
        return;
    }
    uint8_t* const smem = smem_raw + (sbase - raw);  // generic pointer to the aligned base
    SmemCtl& ctl = *reinterpret_cast<SmemCtl*>(smem + kSmemBytes);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const Unit w = decode_unit<PAGED>(a, blockIdx.x);
    if (w.flags && threadIdx.x == 0)
        atomicOr(a.err, w.flags);
    if (!w.valid)
        return;  // uniform over the CTA, before any barrier or allocation
    volatile int* abort = &ctl.abort;

    const bool rope = PAGED && a.rope;
    const int* const trow = PAGED ? a.block_tables + (size_t)w.b * a.max_blocks : nullptr;
    // one contiguous K or V tile into `dst`: a 64 x 128 box per half (the paged
    // form copies page by page, in the producer loop below)
    auto load_tile = [&](const CUtensorMap* map, uint32_t dst, uint32_t bar, int j) {
        for (int h = 0; h < 2; ++h)
            tma_load_4d(dst + h * kBoxBytes, map, bar, h * 64, w.g, j * BN, w.b);
    };
    auto load_q = [&](int t, uint32_t bar) {
        for (int h = 0; h < 2; ++h) {
            const uint32_t dst = sbase + kSmemQ + t * kTileBytes + h * kBoxBytes;
            if (PAGED)
                tma_load_3d(dst, &tmQ, bar, h * 64, w.head[t], w.q_base + w.row0[t]);
            else
                tma_load_4d(dst, &tmQ, bar, h * 64, w.head[t], w.row0[t], w.b);
        }
    };

    // The TMA thread sets up the barriers and sends the first tiles on their way
    // before the set-up barrier (tensor memory is allocated meanwhile): Q_0 and
    // K_0 first, which the first score GEMM needs, then Q_1 and V_0.  Paged K/V
    // wait until after it: their page ids come from global memory, and the
    // other warps would wait for those reads at the barrier.
    constexpr bool kEarlyKV = !PAGED;
    if (warp == kTmaWarp && lane == 0) {
        ctl.abort = 0;
        mbar_init(smem_u32(&ctl.q_full), 1);
        mbar_init(smem_u32(&ctl.q0_full), 1);
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(smem_u32(&ctl.k_full[s]), 1);
            mbar_init(smem_u32(&ctl.k_empty[s]), 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(smem_u32(&ctl.v_full[s]), 1);
            mbar_init(smem_u32(&ctl.v_empty[s]), 1);
        }
        for (int t = 0; t < 2; ++t) {
            // 256 arrivals when both warpgroups rotate rows of both tiles (head pairs)
            mbar_init(smem_u32(&ctl.q_ready[t]), a.head_pairs ? 256 : 128);
            mbar_init(smem_u32(&ctl.s_full[t]), 1);
            // tile 0's P barrier also takes the relay warp's arrival (operands in place)
            mbar_init(smem_u32(&ctl.p_full[t]), t == 0 ? 129 : 128);
            mbar_init(smem_u32(&ctl.o_full[t]), 1);
        }
        mbar_init(smem_u32(&ctl.mma_done), 1);
        fence_mbar_init();
        fence_proxy_async_smem();   // the initialised barriers, before the copies complete on them
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmO);
        const uint32_t qbar = smem_u32(&ctl.q_full);
        const bool q_weight = rope && a.q_w;
        if (rope) {
            // both tiles on one barrier: the softmax warps rotate them in place
            mbar_arrive_expect_tx(qbar, 2 * kTileBytes + (q_weight ? D * 2 : 0));
            if (q_weight)
                bulk_load(sbase + kSmemW, a.q_w, D * 2, qbar);
            load_q(0, qbar);
        } else {
            mbar_arrive_expect_tx(smem_u32(&ctl.q0_full), kTileBytes);
            load_q(0, smem_u32(&ctl.q0_full));
            mbar_arrive_expect_tx(qbar, kTileBytes);
        }
        if (kEarlyKV && w.n_kv > 0 && a.stall_tile != 0) {
            const uint32_t kbar = smem_u32(&ctl.k_full[0]);
            mbar_arrive_expect_tx(kbar, kTileBytes);
            load_tile(&tmK, sbase + kSmemK, kbar, 0);
        }
        load_q(1, qbar);
        if (kEarlyKV && w.n_kv > 0) {
            const uint32_t vbar = smem_u32(&ctl.v_full[0]);
            mbar_arrive_expect_tx(vbar, kTileBytes);
            load_tile(&tmV, sbase + kSmemV, vbar, 0);
        }
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&ctl.tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;
    // Whole warpgroups re-balance registers, each with one setmaxnreg and then only
    // its own code: warps 8-11 (MMA, TMA, relay, idle) down, warps 0-7 (softmax) up.
    if (warp >= 8) {
        regs_decrease<kControlRegs>();
        if (warp == kTmaWarp) {
            // ------------------------------------------------------------ TMA producer
            if (lane == 0) {
                const uint32_t qbar = smem_u32(&ctl.q_full);
                // contiguous: tile 0's K and V went out with the Q tiles
                int n_k = kEarlyKV && w.n_kv > 0 ? 1 : 0, n_v = n_k;  // K / V tiles issued so far
                bool ok = true;
                // paged: a tile is one 64 x 16 box per half and page (a page past
                // the context, or any id outside the cache, reads as zeros); the page
                // ids of the next tile are read while this one's stages are awaited,
                // and serve both its K and its V copies
                int phys[kPagesPerTile];
                auto read_pages = [&](int j) {
#pragma unroll
                    for (int k = 0; k < kPagesPerTile; ++k) {
                        const int p = j * kPagesPerTile + k;
                        phys[k] = p < w.n_pages ? trow[p] : -1;
                    }
                };
                auto load_paged = [&](const CUtensorMap* map, uint32_t dst, uint32_t bar) {
#pragma unroll
                    for (int k = 0; k < kPagesPerTile; ++k)
                        for (int h = 0; h < 2; ++h)
                            tma_load_4d(dst + h * kBoxBytes + k * kPageBoxBytes, map, bar, h * 64, 0, w.g, phys[k]);
                };
                if (PAGED && n_k < w.n_kv)
                    read_pages(n_k);
                for (int j = n_k; j < w.n_kv && ok; ++j) {
                    const int sk = j % kKStages;
                    ok = mbar_wait(smem_u32(&ctl.k_empty[sk]), ((j / kKStages) & 1) ^ 1, abort);
                    if (!ok)
                        break;
                    const uint32_t kbar = smem_u32(&ctl.k_full[sk]);
                    if (j != a.stall_tile) {
                        mbar_arrive_expect_tx(kbar, kTileBytes);
                        if (PAGED)
                            load_paged(&tmK, sbase + kSmemK + sk * kTileBytes, kbar);
                        else
                            load_tile(&tmK, sbase + kSmemK + sk * kTileBytes, kbar, j);
                    }
                    ++n_k;
                    const int sv = j % kVStages;
                    ok = mbar_wait(smem_u32(&ctl.v_empty[sv]), ((j / kVStages) & 1) ^ 1, abort);
                    if (!ok)
                        break;
                    const uint32_t vbar = smem_u32(&ctl.v_full[sv]);
                    mbar_arrive_expect_tx(vbar, kTileBytes);
                    if (PAGED) {
                        load_paged(&tmV, sbase + kSmemV + sv * kTileBytes, vbar);
                        if (j + 1 < w.n_kv)
                            read_pages(j + 1);
                    } else {
                        load_tile(&tmV, sbase + kSmemV + sv * kTileBytes, vbar, j);
                    }
                    ++n_v;
                }
                if (!ok)
                    flag_abort(&ctl, a.err);
                // drain: every copy this CTA started has landed before shared memory
                // is released (bounded by time only, not by the abort flag)
                const int no_abort = 0;
                mbar_wait(qbar, 0, &no_abort);
                if (!rope)
                    mbar_wait(smem_u32(&ctl.q0_full), 0, &no_abort);
                for (int s = 0; s < kKStages; ++s) {
                    // loads issued into stage s: tiles j < n_k with j % kKStages == s,
                    // except a withheld one
                    const int c = (n_k > s ? (n_k - s + kKStages - 1) / kKStages : 0) -
                                  ((a.stall_tile >= 0 && a.stall_tile < n_k && a.stall_tile % kKStages == s) ? 1 : 0);
                    if (c)
                        mbar_wait(smem_u32(&ctl.k_full[s]), (c - 1) & 1, &no_abort);
                }
                for (int s = 0; s < kVStages; ++s) {
                    const int c = n_v > s ? (n_v - s + kVStages - 1) / kVStages : 0;
                    if (c)
                        mbar_wait(smem_u32(&ctl.v_full[s]), (c - 1) & 1, &no_abort);
                }
            }
        } else if (warp == kRelayWarp) {
            // ------------------------------------------------------------ relay warp
            // For each key tile j, once V_j and K_{j+1} have landed it adds the
            // 129th arrival to p_full[0]'s phase j, so the MMA warp checks a single
            // barrier before PV0(j) / S0(j+1).  It waits for phase j-1 to complete
            // first, so that each phase gets exactly one of its arrivals.
            if (lane == 0) {
                bool ok = true;
                for (int j = 0; j < w.n_kv && ok; ++j) {
                    if (j > 0)
                        ok = mbar_wait(smem_u32(&ctl.p_full[0]), (j - 1) & 1, abort);
                    ok = ok && mbar_wait(smem_u32(&ctl.v_full[j % kVStages]), (j / kVStages) & 1, abort);
                    if (ok && j + 1 < w.n_kv)
                        ok = mbar_wait(smem_u32(&ctl.k_full[(j + 1) % kKStages]), ((j + 1) / kKStages) & 1, abort);
                    if (ok)
                        mbar_arrive(smem_u32(&ctl.p_full[0]));
                }
                if (!ok)
                    flag_abort(&ctl, a.err);
            }
        } else if (warp == kMmaWarp) {
            // ------------------------------------------------------------ MMA warp
            // The whole warp follows the schedule (so it can clear shared memory
            // when needed); lane 0 issues the MMAs and commits.
            const bool leader = lane == 0;
            const uint32_t idesc_s = idesc_f16_f32(BM, BN, false, false);
            const uint32_t idesc_o = idesc_f16_f32(BM, D, false, true);
            // descriptors of the first tile of each region; moving within a region
            // only adds (byte offset >> 4) to the start-address field (all shared
            // addresses are below 256 KB, so the 14-bit field cannot overflow)
            const uint64_t dq = sdesc_sw128(sbase + kSmemQ, 16, 1024);
            const uint64_t dk = sdesc_sw128(sbase + kSmemK, 16, 1024);
            const uint64_t dv = sdesc_sw128(sbase + kSmemV, kBoxBytes, 1024);
            auto issue_s = [&](int t, int s) {
                const uint64_t aq = dq + ((t * kTileBytes) >> 4);
                const uint64_t bk = dk + ((s * kTileBytes) >> 4);
    #pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk / 4) * kBoxBytes + (kk % 4) * 32) >> 4;
                    mma_f16_ss(tmem + t * BN, aq + off, bk + off, idesc_s, kk > 0);
                }
            };
            auto issue_o = [&](int t, int s, bool acc) {
                const uint64_t bv = dv + ((s * kTileBytes) >> 4);
    #pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_f16_ts(tmem + 256 + t * D, tmem + t * BN + kk * 8, bv + ((kk * 2048) >> 4),
                               idesc_o, (acc || kk > 0) ? 1u : 0u);
            };
            // The MMA warp sits in back-pressured MMA issue most of a step, so the
            // barriers it checks next are usually complete by then; a complete one
            // costs a non-blocking test here (a try_wait on it cost ~150-300 cycles,
            // during which the tensor pipe's short queue ran dry).
            auto wait = [&](uint64_t& bar, uint32_t parity) -> bool {
                const uint32_t b = smem_u32(&bar);
                if (__all_sync(0xffffffffu, mbar_test(b, parity)))
                    return true;
                return __all_sync(0xffffffffu, mbar_wait(b, parity, abort)) != 0;
            };
            // with the query prologue folded in, each tile's score GEMM waits for its
            // rows to be normalised and rotated (else for its TMA load)
            bool ok = wait(rope ? ctl.q_ready[0] : ctl.q0_full, 0) && wait(ctl.k_full[0], 0);
            if (ok) {
                tc_fence_after();
                if (leader) {
                    issue_s(0, 0);
                    mma_commit(smem_u32(&ctl.s_full[0]));
                }
                __syncwarp();
            }
            ok = ok && wait(rope ? ctl.q_ready[1] : ctl.q_full, 0);
            if (ok) {
                tc_fence_after();
                if (leader) {
                    issue_s(1, 0);
                    mma_commit(smem_u32(&ctl.s_full[1]));
                    mma_commit(smem_u32(&ctl.k_empty[0]));
                }
                __syncwarp();
            }
            for (int j = 0; j < w.n_kv && ok; ++j) {
                const int sv = j % kVStages;
                const int sk1 = (j + 1) % kKStages;
                const bool more = j + 1 < w.n_kv;
                // Operands first (usually long in place: the warp is idle until tile 0's
                // P is ready anyway), so that nothing stands between PV0 and S0 below:
                // each mbarrier wait costs the issuing warp of order a hundred cycles.
                // p_full[0] completes once tile 0's P is written and the relay warp
                // has seen V_j and K_{j+1} land (every barrier test here is a
                // shared-memory access that queues behind the tensor core's operand
                // reads; one test instead of three shortens the gap in which the
                // tensor pipe's short queue runs dry)
                ok = wait(ctl.p_full[0], j & 1);
                if (!ok)
                    break;
                if (PAGED && (j + 1) * BN > w.Lkv) {
                    // Keys from L_kv to the end of the last page are cache slots that may
                    // hold anything (even NaN, and 0 * NaN would reach O through the MMA
                    // although their P is 0): zero those V rows.  Later pages arrive
                    // from TMA as zeros already.
                    const int r0 = w.Lkv - j * BN;
                    const int r1 = min(BN, w.n_pages * kPageSize - j * BN);
                    uint8_t* vt = smem + kSmemV + sv * kTileBytes;
                    for (int idx = lane; idx < (r1 - r0) * 16; idx += 32) {
                        const int rr = r0 + idx / 16, hh = (idx % 16) / 8, c16 = idx % 8;
                        *reinterpret_cast<uint4*>(vt + hh * kBoxBytes + rr * 128 + c16 * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                tc_fence_after();
                if (leader) {
                    issue_o(0, sv, j > 0);
                    if (!more)
                        mma_commit(smem_u32(&ctl.o_full[0]));
                    else {
                        issue_s(0, sk1);
                        mma_commit(smem_u32(&ctl.s_full[0]));
                    }
                }
                __syncwarp();
                ok = wait(ctl.p_full[1], j & 1);
                if (!ok)
                    break;
                tc_fence_after();
                if (leader) {
                    issue_o(1, sv, j > 0);
                    mma_commit(smem_u32(&ctl.v_empty[sv]));
                    if (!more)
                        mma_commit(smem_u32(&ctl.o_full[1]));
                    if (more) {
                        issue_s(1, sk1);
                        mma_commit(smem_u32(&ctl.s_full[1]));
                        mma_commit(smem_u32(&ctl.k_empty[sk1]));
                    }
                }
                __syncwarp();
            }
            if (leader) {
                if (!ok)
                    flag_abort(&ctl, a.err);
                // drain: all MMAs issued by this thread are complete before TMEM is released
                const int no_abort = 0;
                mma_commit(smem_u32(&ctl.mma_done));
                mbar_wait(smem_u32(&ctl.mma_done), 0, &no_abort);
            }
        }
    } else {
        regs_increase<kSoftmaxRegs>();
        // ------------------------------------------------------------ softmax warps
        const int t = warp / 4;             // Q tile
        const int quad = warp % 4;          // TMEM lane quadrant = rows [32*quad, +32)
        const int row = quad * 32 + lane;   // row within the tile = TMEM lane
        const int my_row0 = t ? w.row0[1] : w.row0[0];
        const int my_head = t ? w.head[1] : w.head[0];
        const int q_row = my_row0 + row;    // query row within the sequence (chunk)
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_addr + t * BN;
        const uint32_t tO = tmem + lane_addr + 256 + t * D;
        const float c = a.scale_log2;
        // keys [0, key_end) are visible to this row: up to its own position
        // (off + q_row) with the causal mask, else the whole context
        const int key_end = a.causal ? min(w.off + q_row + 1, w.Lkv) : w.Lkv;
        float m_ref = -CUDART_INF_F;  // reference max (log2 units) shared by l and O
        float l_sum = 0.f;
        bool ok = true;
        if (PAGED && a.rope) {
            // Query prologue (norm_rope_one).  Rows past the chunk are left as
            // loaded (their output is not stored); a row whose position lies
            // outside the table is left unrotated and flagged.  The table entries
            // are fetched while the tiles are still in flight.
            const bool norm = a.q_w != nullptr;
            auto run = [&](auto shared_tag) -> bool {
                constexpr bool kShared = decltype(shared_tag)::value;   // the tiles' rows share positions
                constexpr int kPasses = kShared ? 4 : 8;
                float4 cs[kPasses][4];
                uint32_t rotate = 0;   // bit p (+ 8 for tile 1 when shared): rotate this lane's row of pass p
                bool bad_pos = false;
#pragma unroll
                for (int p = 0; p < kPasses; ++p) {
                    const int r = rope_row(kShared, t, p, quad, lane);
#pragma unroll
                    for (int tt = 0; tt < 2; ++tt) {
                        if (kShared || tt == t) {
                            const int qr_row = w.row0[tt] + r;
                            const int pos = w.off + qr_row;
                            if (qr_row < w.Lq) {
                                if (pos >= 0 && pos < a.max_pos)
                                    rotate |= 1u << (p + 8 * tt);
                                else
                                    bad_pos = true;
                            }
                        }
                    }
                    const int pos = w.off + (kShared ? w.row0[0] : my_row0) + r;
                    const bool in_table = pos >= 0 && pos < a.max_pos;
                    const float4* trow = a.rope_table + (size_t)(in_table ? pos : 0) * 32 + lane % 8;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        cs[p][i] = __ldg(trow + i * 8);
                }
                if (__any_sync(0xffffffffu, bad_pos) && lane == 0)
                    atomicOr(a.err, kDevErrBadPosition);
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl.q_full), 0, abort)))
                    return false;
                uint4 wlo = make_uint4(0u, 0u, 0u, 0u), whi = wlo;
                if (norm) {
                    const uint4* wsm = reinterpret_cast<const uint4*>(smem + kSmemW);
                    wlo = wsm[lane % 8];
                    whi = wsm[8 + lane % 8];
                }
                // batches of rows per lane: shared, 2 passes x both tiles; own tile,
                // 2 passes (its 8 passes' table entries already hold 128 registers)
                constexpr int kBatch = kShared ? 4 : 2;
#pragma unroll
                for (int b = 0; b < 8 / kBatch; ++b) {   // 8 rows per lane either way
                    int row[kBatch], tile[kBatch], pass[kBatch];
                    uint32_t store = 0;
#pragma unroll
                    for (int n = 0; n < kBatch; ++n) {
                        pass[n] = kShared ? 2 * b + n / 2 : kBatch * b + n;
                        tile[n] = kShared ? n % 2 : t;
                        row[n] = rope_row(kShared, t, pass[n], quad, lane);
                        store |= (rotate >> (pass[n] + 8 * tile[n]) & 1u) << n;
                    }
                    norm_rope_batch(smem + kSmemQ, row, tile, pass, cs, store, wlo, whi, norm, a.eps, lane);
                }
                return true;
            };
            const bool shared = a.head_pairs;
            if (shared ? run(std::true_type{}) : run(std::false_type{})) {
                fence_proxy_async_smem();   // the score GEMMs read these rows through the async proxy
                // both tiles' barriers when the rows are shared, else the own tile's
                if (shared || t == 0)
                    mbar_arrive(smem_u32(&ctl.q_ready[0]));
                if (shared || t == 1)
                    mbar_arrive(smem_u32(&ctl.q_ready[1]));
            } else {
                flag_abort(&ctl, a.err);   // every wait below now gives up at once
            }
        }
        for (int j = 0; j < w.n_kv; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl.s_full[t]), j & 1, abort));
            if (!ok)
                break;
            tc_fence_after();
            const int limit = key_end - j * BN;
            const bool masked = __any_sync(0xffffffffu, limit < BN);
            uint32_t sr[4][32];
            float rs[8];
            auto load_s = [&]() {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    tmem_ld32(tS + q4 * 32, sr[q4]);
                tmem_ld_wait();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    reg_fence32(sr[q4]);
                if (masked) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (q4 * 32 + i >= limit)
                                sr[q4][i] = __float_as_uint(-CUDART_INF_F);
                }
            };
            // move the reference to the tile's row max if it exceeds it by more than
            // the threshold (always on the first tile, whose reference is -inf)
            bool grow = false;
            float alpha = 1.f;
            auto move_ref = [&](float mx) {
                const float m_new = fmaxf(m_ref, mx * c);
                if (m_new > m_ref + kRescaleThreshold) {
                    grow = true;
                    alpha = ex2_approx(m_ref - m_new);
                    m_ref = m_new;
                    l_sum *= alpha;
                }
            };
            load_s();
            if (j == 0)
                move_ref(fmaxf(fmax3(max32(sr[0]), max32(sr[1]), max32(sr[2])), max32(sr[3])));
            // One straight pass against the current reference.  Every p of the row is
            // at most the row's sum, so a sum within 2^threshold proves that no p
            // exceeds it and the reference holds; only otherwise is the tile's max
            // taken (from S, still intact in TMEM) to decide.
#pragma unroll
            for (int k8 = 0; k8 < 8; ++k8)
                rs[k8] = 0.f;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
                exp_pack32(sr[q4], c, -m_ref, rs);
            fadd2(rs[0], rs[1], rs[2], rs[3]);
            fadd2(rs[4], rs[5], rs[6], rs[7]);
            fadd2(rs[0], rs[1], rs[4], rs[5]);
            float tile_sum = rs[0] + rs[1];
            if (j > 0 && __any_sync(0xffffffffu, tile_sum > kSumLimit)) {
                // rare: reload S, move the reference if the max grew past the
                // threshold, and redo the pass (the same values if it did not)
                load_s();
                move_ref(fmaxf(fmax3(max32(sr[0]), max32(sr[1]), max32(sr[2])), max32(sr[3])));
#pragma unroll
                for (int k8 = 0; k8 < 8; ++k8)
                    rs[k8] = 0.f;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    exp_pack32(sr[q4], c, -m_ref, rs);
                fadd2(rs[0], rs[1], rs[2], rs[3]);
                fadd2(rs[4], rs[5], rs[6], rs[7]);
                fadd2(rs[0], rs[1], rs[4], rs[5]);
                tile_sum = rs[0] + rs[1];
            }
            // S has been read for the last time: P overwrites its first 64 columns
            tmem_st32_even(tS, sr[0], sr[1]);
            tmem_st32_even(tS + 32, sr[2], sr[3]);
            l_sum += tile_sum;
            if (j > 0 && __any_sync(0xffffffffu, grow)) {
                // O_t holds the previous tiles' sum (its last PV completed before
                // s_full fired and the next PV waits for p_full): bring it to the
                // new reference max
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t orr[32];
                    tmem_ld32(tO + q4 * 32, orr);
                    tmem_ld_wait();
                    reg_fence32(orr);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
                    tmem_st32(tO + q4 * 32, orr);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(smem_u32(&ctl.p_full[t]));
        }
        if (ok)
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl.o_full[t]), 0, abort));
        if (!ok) {
            flag_abort(&ctl, a.err);
        } else {
            tc_fence_after();
            const float inv = 1.f / l_sum;
            // A whole tile leaves through shared memory and TMA stores: Q_t's
            // buffer is free (every S GEMM that read it completed before o_full),
            // each thread writes its row there in the 128-byte swizzled layout of
            // the O tensor map's boxes (conflict-free: 8 consecutive rows cover all
            // 16-byte bank groups), and each warp stores its 32 rows (two 64-dim
            // boxes of 32 rows).  A tile that runs past the end of the sequence
            // (chunk) stores its rows one by one.
            const bool whole = my_row0 + BM <= w.Lq;   // uniform over the warpgroup
            const bool store = q_row < w.Lq;
            __half* dst = a.O + ((size_t)(w.q_base + q_row) * a.H_q + my_head) * D;
            uint8_t* const stile = smem + kSmemQ + t * kTileBytes;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t orr[32];
                tmem_ld32(tO + q4 * 32, orr);
                tmem_ld_wait();
                reg_fence32(orr);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    uint4 pk;
                    pk.x = pack_half2(__uint_as_float(orr[8 * v + 0]) * inv, __uint_as_float(orr[8 * v + 1]) * inv);
                    pk.y = pack_half2(__uint_as_float(orr[8 * v + 2]) * inv, __uint_as_float(orr[8 * v + 3]) * inv);
                    pk.z = pack_half2(__uint_as_float(orr[8 * v + 4]) * inv, __uint_as_float(orr[8 * v + 5]) * inv);
                    pk.w = pack_half2(__uint_as_float(orr[8 * v + 6]) * inv, __uint_as_float(orr[8 * v + 7]) * inv);
                    if (whole) {
                        const int c16 = q4 * 4 + v;   // 16-byte chunk of the 256-byte row
                        *reinterpret_cast<uint4*>(stile + (c16 / 8) * kBoxBytes + row * 128 +
                                                  (((c16 % 8) ^ (row % 8)) << 4)) = pk;
                    } else if (store) {
                        *reinterpret_cast<uint4*>(dst + q4 * 32 + v * 8) = pk;
                    }
                }
            }
            if (whole) {
                // each warp stores its own 32 rows (1024-byte aligned inside the
                // tile, so the swizzle phase is the tile's) once they are written
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const uint32_t src = sbase + kSmemQ + t * kTileBytes + quad * 32 * 128;
                    const int r0 = my_row0 + quad * 32;
                    for (int h = 0; h < 2; ++h) {
                        if (PAGED)
                            tma_store_3d(&tmO, src + h * kBoxBytes, h * 64, my_head, w.q_base + r0);
                        else
                            tma_store_4d(&tmO, src + h * kBoxBytes, h * 64, my_head, r0, w.b);
                    }
                    bulk_commit_group();
                    bulk_wait_group_read0();   // shared memory stays valid until read
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp)
        tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// FP16 tensor map, 128-byte swizzle, zero fill out of bounds.  dims/strides
// innermost first (strides in bytes, for dims 1..rank-1).
bool make_map(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims,
              const cuuint64_t* strides, const cuuint32_t* box)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, rank, const_cast<void*>(ptr), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// [B,S,H,128]: boxes of 64 head-dim x 1 head x `rows` rows (128 for loads, 32
// for the per-warp O stores) x 1 batch.
bool make_bshd_map(CUtensorMap* m, const void* ptr, int B, int S, int H, int rows = BM)
{
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2,
                                   (cuuint64_t)S * H * D * 2};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
    return make_map(m, ptr, 4, dims, strides, box);
}

// packed [total, H, 128]: boxes of 64 head-dim x 1 head x `rows` rows.
bool make_packed_map(CUtensorMap* m, const void* ptr, int total, int H, int rows = BM)
{
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)total};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)rows};
    return make_map(m, ptr, 3, dims, strides, box);
}

// paged cache [num_blocks, H_kv, 16, 128]: boxes of 64 head-dim x 16 slots (one page).
bool make_cache_map(CUtensorMap* m, const void* ptr, long long num_blocks, int H_kv)
{
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)kPageSize, (cuuint64_t)H_kv,
                                (cuuint64_t)num_blocks};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)kPageSize * D * 2,
                                   (cuuint64_t)H_kv * kPageSize * D * 2};
    const cuuint32_t box[4] = {64, kPageSize, 1, 1};
    return make_map(m, ptr, 4, dims, strides, box);
}

// the shared-memory opt-in is a per-context, per-kernel attribute: set once per
// device and context (a context that replaced one after a reset gets it too)
template <bool PAGED>
cudaError_t ensure_smem_attr()
{
    static std::mutex mtx;
    static unsigned long long done_ctx[64] = {};   // context the attribute was set in
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
    std::lock_guard<std::mutex> lock(mtx);
    if (done_ctx[dev] != ctx) {
        cudaFuncAttributes fa{};
        e = cudaFuncGetAttributes(&fa, prefill_kernel<PAGED>);
        if (e != cudaSuccess)
            return e;
        // the warpgroups' register re-balance must fit the pool the CTA launches with
        if ((long long)fa.numRegs * kThreads < 256LL * kSoftmaxRegs + 128LL * kControlRegs)
            return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(prefill_kernel<PAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemAlloc);
        if (e != cudaSuccess)
            return e;
        done_ctx[dev] = ctx;
    }
    return cudaSuccess;
}

// (batch, kv head) groups per super-group of the unit order: as many as keep
// their K and V (2 * keys * 256 bytes each, keys bounded by max_keys) within
// about a quarter of the 129 MB L2.
int groups_per_super(int n_groups, long long max_keys)
{
    constexpr long long kBudget = 32ll << 20;
    const long long per_group = 2 * max_keys * D * 2;
    const long long g = per_group > 0 ? kBudget / per_group : n_groups;
    return (int)(g < 1 ? 1 : (g > n_groups ? n_groups : g));
}

void fill_common(PrefillArgs& a, int B, int H_q, int H_kv, int rows, int causal)
{
    a.B = B;
    a.H_q = H_q;
    a.H_kv = H_kv;
    a.group = H_q / H_kv;
    a.head_pairs = (a.group % 2 == 0) ? 1 : 0;
    const int pairs_per_g = a.head_pairs ? a.group / 2 : a.group;
    a.n_mb = a.head_pairs ? (rows + BM - 1) / BM : (rows + 2 * BM - 1) / (2 * BM);
    a.units_per_mb = B * H_kv * pairs_per_g;
    a.groups_per_super = B * H_kv;   // one super-group unless the caller sizes them
    a.causal = causal ? 1 : 0;
    a.scale_log2 = kLog2e / sqrtf((float)D);
    a.stall_tile = -1;
}

}  // namespace

cudaError_t launch_prefill(const void* Q, const void* K, const void* V, void* O, int B, int S,
                           int H_q, int H_kv, int causal, int stall_tile, cudaStream_t stream)
{
    cudaError_t e = ensure_smem_attr<false>();
    if (e != cudaSuccess)
        return e;
    CUtensorMap mq, mk, mv, mo;
    if (!make_bshd_map(&mq, Q, B, S, H_q) || !make_bshd_map(&mk, K, B, S, H_kv) ||
        !make_bshd_map(&mv, V, B, S, H_kv) || !make_bshd_map(&mo, O, B, S, H_q, 32))
        return cudaErrorInvalidValue;
    PrefillArgs a{};
    a.O = static_cast<__half*>(O);
    a.err = device_error_word();
    if (!a.err)
        return cudaErrorInvalidSymbol;
    fill_common(a, B, H_q, H_kv, S, causal);
    a.groups_per_super = groups_per_super(B * H_kv, (long long)S);
    a.S = S;
    a.stall_tile = stall_tile;
    const long long grid = (long long)a.units_per_mb * a.n_mb;
    if (grid > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    prefill_kernel<false><<<(unsigned)grid, kThreads, kSmemAlloc, stream>>>(mq, mk, mv, mo, a);
    return cudaGetLastError();
}

cudaError_t launch_prefill_paged(const void* Q, const void* k_cache, const void* v_cache, void* O,
                                 const int* cu_seqlens_q, const int* seq_lens_kv,
                                 const int* block_tables, int B, int max_seqlen_q, int total_q,
                                 int H_q, int H_kv, int max_blocks_per_seq, long long num_blocks,
                                 int causal, const QueryPrologue* qp, cudaStream_t stream)
{
    cudaError_t e = ensure_smem_attr<true>();
    if (e != cudaSuccess)
        return e;
    CUtensorMap mq, mk, mv, mo;
    if (!make_packed_map(&mq, Q, total_q, H_q) || !make_cache_map(&mk, k_cache, num_blocks, H_kv) ||
        !make_cache_map(&mv, v_cache, num_blocks, H_kv) || !make_packed_map(&mo, O, total_q, H_q, 32))
        return cudaErrorInvalidValue;
    PrefillArgs a{};
    a.O = static_cast<__half*>(O);
    a.err = device_error_word();
    if (!a.err)
        return cudaErrorInvalidSymbol;
    fill_common(a, B, H_q, H_kv, max_seqlen_q, causal);
    a.groups_per_super = groups_per_super(B * H_kv, (long long)max_blocks_per_seq * kPageSize);
    a.S = 0;
    a.cu_q = cu_seqlens_q;
    a.seq_lens_kv = seq_lens_kv;
    a.block_tables = block_tables;
    a.max_blocks = max_blocks_per_seq;
    a.total_q = total_q;
    if (qp) {
        a.rope = 1;
        a.q_w = static_cast<const __half*>(qp->q_weight);
        a.rope_table = reinterpret_cast<const float4*>(qp->cos_sin);
        a.max_pos = qp->max_pos;
        a.eps = qp->eps;
    }
    const long long grid = (long long)a.units_per_mb * a.n_mb;
    if (grid > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    prefill_kernel<true><<<(unsigned)grid, kThreads, kSmemAlloc, stream>>>(mq, mk, mv, mo, a);
    return cudaGetLastError();
}

}  // namespace attn
