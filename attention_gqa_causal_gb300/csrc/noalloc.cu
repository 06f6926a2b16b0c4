// noalloc.cu -- paged decode that allocates nothing: the split-K scratch lives
// in a fixed buffer compiled into the library.
//
// Some callers cannot call cudaMalloc: code hosted inside another runtime
// that owns every byte of device memory and hands out no allocator, programs
// that run under a fixed, pre-accounted memory budget, and latency-critical
// loops that must not risk the device-wide synchronisation that cudaMalloc
// and cudaFree can cause.  attn_decode_paged would grow a library-owned
// buffer for them, and attn_decode_paged_ws needs a buffer they cannot make.
// This entry point instead uses kScratchBytes of scratch that exists once the
// library's device code is loaded on a GPU and stays there, on every GPU that
// loads it, until the process exits.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "attn.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB
static_assert(kScratchBytes == ATTN_NOALLOC_SCRATCH_BYTES, "header and library disagree");

// The split-K partials (O and log-sum-exp per split) of one call.  Host code
// must not use this name as a pointer: on the host it only stands for the
// symbol, so its device address is looked up with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
// Set-up per device: the device address of g_scratch, and the context it
// belongs to.  A device whose context was replaced (cudaDeviceReset) has its
// module loaded anew, possibly at another address, so the set-up runs again.
struct ScratchSlot {
    unsigned long long ctx = 0;
    void* addr = nullptr;
};
ScratchSlot g_slot[kMaxDevices];

// Device address of g_scratch on the current device.  cudaGetSymbolAddress
// runs once per device and context (the first call on a device, and the
// first after its context was replaced); later calls reuse the address.
cudaError_t scratch_address(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    unsigned long long ctx = 0;
    e = attn::current_context_id(&ctx);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lock(g_mutex);
    ScratchSlot& s = g_slot[dev];
    if (!s.addr || s.ctx != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess)
            return e;
        s.addr = p;
        s.ctx = ctx;
    }
    *out = s.addr;
    return cudaSuccess;
}

}  // namespace

extern "C" ATTN_API int attn_decode_paged_noalloc(const void* q, const void* k_cache,
                                                  const void* v_cache, void* out,
                                                  const int* block_tables, const int* seq_lens,
                                                  int num_seqs, int H_q, int H_kv, int D,
                                                  int max_blocks_per_seq, int block_size,
                                                  cudaStream_t stream)
{
    // The scratch size is checked first, so a problem that does not fit is
    // refused before anything is launched.  Invalid sizes give need == 0 and
    // are reported by the argument checks of attn_decode_paged_ws.
    const size_t need = attn_decode_paged_workspace_bytes(num_seqs, H_q, H_kv, D,
                                                          max_blocks_per_seq, block_size, 0);
    if (need > kScratchBytes)
        return ATTN_ERR_WORKSPACE;
    if (num_seqs == 0 || need == 0)
        return attn_decode_paged_ws(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs,
                                    H_q, H_kv, D, max_blocks_per_seq, block_size, 0, nullptr, 0,
                                    stream);
    void* scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess)
        return attn::record_cuda_error(e);
    // Every partial the combine step reads is written earlier in this same
    // call, so nothing a previous call left in the buffer is ever read and
    // nothing needs clearing.
    return attn_decode_paged_ws(q, k_cache, v_cache, out, block_tables, seq_lens, num_seqs, H_q,
                                H_kv, D, max_blocks_per_seq, block_size, 0, scratch,
                                kScratchBytes, stream);
}
