// prefill_noalloc.cu -- kda_prefill_noalloc: the chunked prefill for callers
// that cannot allocate device memory.
//
// Some callers have no allocator to hand the library a workspace: code running
// inside a framework that owns every device allocation, an embedded runtime
// that forbids cudaMalloc after start-up, or a host path that must never block
// on the allocator.  For them the workspace lives in a fixed file-scope device
// array instead.  Its size is a hard limit: every GPU that loads this library
// keeps the array resident until the process exits, so it is kept modest.
//
// Host code may not pass the array's name to a kernel (on the host that name is
// a stand-in, not a device address); the device address is fetched once per
// device with cudaGetSymbolAddress, with that device current, on the first call
// made on it, and cached.  That first call therefore performs a runtime query
// and should be made before any stream capture begins.
//
// Every call shares the one array, and the array keeps whatever the previous
// call left in it.  The only part that must start at zero, the device status
// word, is cleared by the prefill itself at the start of each call; the
// per-call sequence table and handoff are fully rewritten.  Calls whose work
// can overlap on the GPU (different streams, different host threads) race on
// the array: they must be ordered by the caller.
#include <mutex>

#include "kda_common.cuh"

namespace {

constexpr size_t kScratchBytes = (size_t)KDA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_setup_lock;
void *g_scratch_ptr[kMaxDevices];

// Device address of g_noalloc_scratch on the current device, looked up once.
cudaError_t scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> guard(g_setup_lock);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" kda_status kda_prefill_noalloc(const void *q, const void *k, const void *v,
                                          const float *g, const float *beta,
                                          const float *init_state, const int32_t *cu_seqlens,
                                          void *out, float *final_state, float *ckpts,
                                          const kda_prefill_desc *desc, kda_stream_t stream)
{
    size_t need = 0;
    const kda_status ds = kda::prefill_workspace_bytes(desc, &need);   // sets the message on error
    if (ds != KDA_OK) return ds;
    if (need > kScratchBytes) {
        return kda::fail_with_message(KDA_ERR_UNSUPPORTED,
                                      "kda_prefill_noalloc: this call needs %zu bytes of scratch, more than the "
                                      "built-in %zu; use kda_prefill with a caller workspace",
                                      need, kScratchBytes);
    }
    void *scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess)
        return kda::fail_with_message(KDA_ERR_CUDA, "kda_prefill_noalloc: scratch address: %s",
                                      cudaGetErrorString(e));
    return kda::prefill_call(q, k, v, g, beta, init_state, cu_seqlens, out, final_state, ckpts, desc,
                             scratch, kScratchBytes, stream, false);
}
