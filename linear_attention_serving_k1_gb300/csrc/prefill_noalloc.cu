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
#include <stdint.h>

#include <mutex>

#include "kda_common.cuh"

namespace {

constexpr size_t kScratchBytes = (size_t)KDA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_setup_lock;
void *g_scratch_ptr[kMaxDevices];

// Workspace bytes of `d` with segment_chunks = G (SIZE_MAX if the descriptor
// is then refused).
size_t bytes_with_segments(kda_prefill_desc d, int64_t G)
{
    d.segment_chunks = (int32_t)G;
    size_t b = 0;
    return kda::prefill_workspace_bytes(&d, &b) == KDA_OK ? b : SIZE_MAX;
}

// The automatic segment plan of the tensor-core path may need more than the
// array while a plan of shorter segments fits; the results are the same for
// every segment length, so `d` takes the longest segments that fit: one
// segment when all records fit, else the largest G whose two ring slots and
// fp32 carry fit (their bytes grow with G below the sequence's chunk count).
// Returns the bytes of the plan chosen (of the automatic one if none fits).
size_t fit_segments(kda_prefill_desc *d, size_t need)
{
    if (need <= kScratchBytes || d->segment_chunks != 0 || !kda::use_tc_path(d->dtype, d->head_dim_k, d->chunk))
        return need;
    const int64_t T = d->total_tokens;
    const int64_t len = d->max_seq_len > 0 && d->max_seq_len < T ? d->max_seq_len : T;
    const int64_t maxc = (len + d->chunk - 1) / d->chunk;
    if (maxc <= 1 || maxc > INT32_MAX) return need;
    if (bytes_with_segments(*d, maxc) <= kScratchBytes) {
        d->segment_chunks = (int32_t)maxc;
        return bytes_with_segments(*d, maxc);
    }
    int64_t lo = 0, hi = maxc - 1;   // largest G in [1, maxc - 1] that fits, 0 if none
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) / 2;
        if (bytes_with_segments(*d, mid) <= kScratchBytes) lo = mid;
        else hi = mid - 1;
    }
    if (lo < 1) return need;
    d->segment_chunks = (int32_t)lo;
    return bytes_with_segments(*d, lo);
}

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
    kda_prefill_desc d = *desc;
    need = fit_segments(&d, need);
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
    return kda::prefill_call(q, k, v, g, beta, init_state, cu_seqlens, out, final_state, ckpts, &d,
                             scratch, kScratchBytes, stream, false);
}
