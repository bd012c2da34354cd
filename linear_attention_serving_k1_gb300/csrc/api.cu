// api.cu -- the C ABI declared in include/kda.h: argument validation,
// workspace layout and kernel dispatch.  No allocation, no synchronisation
// (except kda_prefill_status, documented as synchronising, and every call of
// the debug build, which waits for its work to read the index checks).
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <string>

#include <nvtx3/nvToolsExt.h>

#include "kda_common.cuh"

namespace {

// An NVTX range around one entry point (visible in a timeline profiler;
// without a tool attached the calls return at once).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

thread_local std::string g_last_error;

kda_status fail(kda_status s, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

kda_status cuda_fail(cudaError_t e, const char *where)
{
    return fail(KDA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Rows by which the debug build's checks take the token-row buffers to be
// shorter than the call says (KDA_DEBUG_CLIP_TOKENS; 0 in the release build).
int64_t debug_clip_tokens()
{
#ifdef KDA_DEBUG
    if (const char *e = getenv("KDA_DEBUG_CLIP_TOKENS")) {
        const long long n = strtoll(e, nullptr, 10);
        return n > 0 ? (int64_t)n : 0;
    }
#endif
    return 0;
}

const char *dbg_site_name(int32_t site)
{
    switch (site) {
    case kda::kDbgTokenRow: return "token row";
    case kda::kDbgRecord: return "K1 -> K2 record";
    case kda::kDbgState: return "state block";
    case kda::kDbgCkpt: return "checkpoint block";
    default: return "index";
    }
}

// Debug build: once the call's work on `stream` is done, the first index
// check that failed in it (KDA_ERR_BOUNDS); `s` otherwise, and always in the
// release build or while the stream is being captured.
kda_status debug_finish(kda_status s, cudaStream_t stream)
{
    if (!kda::kDebug || s != KDA_OK) return s;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return s;
    }
    if (cs != cudaStreamCaptureStatusNone) return s;
    const cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "debug build: waiting for the call");
    const kda::DbgWord words[] = {kda::dbg_take_prefill_tc(), kda::dbg_take_prefill_simt(), kda::dbg_take_decode()};
    for (const kda::DbgWord &w : words)
        if (w.code != 0)
            return fail(KDA_ERR_BOUNDS, "debug build: %s index %lld outside [0, %lld); the access was skipped",
                        dbg_site_name(w.site), (long long)w.index, (long long)w.extent);
    return s;
}

struct Layout {
    size_t status, cu, chunk_off, ckpt_off, handoff, carry, total;
    int max_chunks;
    kda::SegPlan plan;
};

// Validates the descriptor; fills the workspace layout on success.
kda_status check_desc(const kda_prefill_desc *d, Layout *lay)
{
    if (!d) return fail(KDA_ERR_INVALID_ARG, "desc is NULL");
    if (d->num_seqs < 1) return fail(KDA_ERR_INVALID_ARG, "num_seqs must be >= 1 (got %d)", d->num_seqs);
    if (d->total_tokens < 0) return fail(KDA_ERR_INVALID_ARG, "total_tokens must be >= 0");
    if (d->total_tokens > (int64_t)INT32_MAX / 2)
        return fail(KDA_ERR_UNSUPPORTED, "total_tokens %lld too large", (long long)d->total_tokens);
    if (d->num_heads < 1) return fail(KDA_ERR_INVALID_ARG, "num_heads must be >= 1");
    if (d->head_dim_k != d->head_dim_v)
        return fail(KDA_ERR_UNSUPPORTED, "head_dim_k (%d) != head_dim_v (%d)", d->head_dim_k, d->head_dim_v);
    if (d->head_dim_k != 64 && d->head_dim_k != 128)
        return fail(KDA_ERR_UNSUPPORTED, "head dim %d not in {64, 128}", d->head_dim_k);
    if (d->dtype != KDA_DTYPE_BF16 && d->dtype != KDA_DTYPE_FP32)
        return fail(KDA_ERR_INVALID_ARG, "unknown dtype %d", (int)d->dtype);
    if (d->chunk != 64) return fail(KDA_ERR_UNSUPPORTED, "chunk %d not supported (64)", d->chunk);
    if (d->ckpt_stride < 0 || (d->ckpt_stride > 0 && d->ckpt_stride % d->chunk != 0))
        return fail(KDA_ERR_INVALID_ARG, "ckpt_stride %d must be 0 or a positive multiple of chunk", d->ckpt_stride);
    if (d->ckpt_capacity < 0) return fail(KDA_ERR_INVALID_ARG, "ckpt_capacity must be >= 0");
    if (d->max_seq_len < 0) return fail(KDA_ERR_INVALID_ARG, "max_seq_len must be >= 0");
    if (d->segment_chunks < 0) return fail(KDA_ERR_INVALID_ARG, "segment_chunks must be >= 0");
    if (d->recurrence_ctas < 0) return fail(KDA_ERR_INVALID_ARG, "recurrence_ctas must be >= 0");
    if (d->conv_width < 0 || d->conv_width > kda::kConvTaps)
        return fail(KDA_ERR_UNSUPPORTED, "conv_width %d not in [0, %d]", d->conv_width, kda::kConvTaps);
    if (d->conv_silu != 0 && d->conv_silu != 1)
        return fail(KDA_ERR_INVALID_ARG, "conv_silu must be 0 or 1 (got %d)", d->conv_silu);
    if (d->scalar_gate != 0 && d->scalar_gate != 1)
        return fail(KDA_ERR_INVALID_ARG, "scalar_gate must be 0 or 1 (got %d)", d->scalar_gate);
    const int64_t maxc = d->total_tokens / d->chunk + d->num_seqs;
    if (maxc * d->num_heads > INT32_MAX) return fail(KDA_ERR_UNSUPPORTED, "too many chunks x heads");
    Layout L;
    L.max_chunks = (int)maxc;
    size_t off = 0;
    L.status = off; off = align256(off + sizeof(kda::DevStatus));
    L.cu = off; off = align256(off + sizeof(int32_t) * (size_t)(d->num_seqs + 1));
    L.chunk_off = off; off = align256(off + sizeof(int32_t) * (size_t)(d->num_seqs + 1));
    L.ckpt_off = off; off = align256(off + sizeof(int32_t) * (size_t)(d->num_seqs + 1));
    L.handoff = off;
    L.plan = kda::SegPlan{0, 1, 1, 0, {}};
    if (kda::use_tc_path(d->dtype, d->head_dim_k, d->chunk)) {
        L.plan = kda::tc_segment_plan(d);
        if ((int64_t)d->num_seqs * L.plan.G * d->num_heads > INT32_MAX)
            return fail(KDA_ERR_UNSUPPORTED, "num_seqs x segment_chunks x num_heads too large");
        const size_t rec = kda::tc_handoff_bytes_per_chunk();
        if (L.plan.nseg == 1) {   // every chunk's record, indexed by global chunk
            off = align256(off + rec * (size_t)maxc * (size_t)d->num_heads);
        } else {                  // R ring slots of N x G x H records, then the carry
            off = align256(off + rec * (size_t)L.plan.R * (size_t)d->num_seqs * (size_t)L.plan.G *
                                     (size_t)d->num_heads);
            L.carry = off;
            off = align256(off + sizeof(float) * (size_t)d->num_seqs * (size_t)d->num_heads *
                                     (size_t)d->head_dim_k * (size_t)d->head_dim_v);
        }
    } else {
        const size_t rec = kda::simt_handoff_bytes_per_chunk(d->head_dim_k, d->chunk);
        off = align256(off + rec * (size_t)maxc * (size_t)d->num_heads);
    }
    if (L.plan.nseg == 1) L.carry = off;
    L.total = off;
    *lay = L;
    return KDA_OK;
}

}  // namespace

namespace kda {

kda_status prefill_workspace_bytes(const kda_prefill_desc *desc, size_t *bytes)
{
    Layout L;
    const kda_status s = check_desc(desc, &L);
    if (s == KDA_OK) *bytes = L.total;
    return s;
}

kda_status fail_with_message(kda_status s, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

}  // namespace kda

extern "C" {

const char *kda_last_error(void) { return g_last_error.c_str(); }

int32_t kda_version(void) { return 100; }

size_t kda_prefill_workspace_size(const kda_prefill_desc *desc)
{
    Layout L;
    if (check_desc(desc, &L) != KDA_OK) return 0;
    return L.total;
}

int32_t kda_prefill_launch_count(const kda_prefill_desc *desc)
{
    Layout L;
    if (check_desc(desc, &L) != KDA_OK) return -1;
    return L.plan.nseg > 1 ? 1 + 2 * L.plan.nseg : 3;
}

}  // extern "C"

namespace kda {
kda_status prefill_call(const void *q, const void *k, const void *v, const float *g, const float *beta,
                        const float *init_state, const int32_t *cu_seqlens, void *out, float *final_state,
                        float *ckpts, const kda_prefill_desc *desc, void *workspace, size_t workspace_bytes,
                        kda_stream_t stream, bool use_graph, const PoolArgs *pool, const FusedArgs *fused)
{
    Layout L;
    kda_status s = check_desc(desc, &L);
    if (s != KDA_OK) return s;
    const int64_t T = desc->total_tokens;
    if (T > 0 && (!q || !k || !v || !g || !beta || !out))
        return fail(KDA_ERR_INVALID_ARG, "q, k, v, g, beta and out must be non-NULL");
    if (!cu_seqlens && T % desc->num_seqs != 0)
        return fail(KDA_ERR_INVALID_ARG, "total_tokens %lld not a multiple of num_seqs %d (cu_seqlens NULL)",
                    (long long)T, desc->num_seqs);
    if (pool) {
        if (pool->slots < 0) return fail(KDA_ERR_INVALID_ARG, "pool_slots must be >= 0");
        if (!pool->pool && (pool->init_slots || pool->final_slots || pool->ckpt_slots))
            return fail(KDA_ERR_INVALID_ARG, "state_pool is NULL but a slot table is given");
        if (desc->ckpt_stride > 0 && desc->ckpt_capacity > 0 && !pool->ckpt_slots)
            return fail(KDA_ERR_INVALID_ARG, "ckpt_slots is NULL but ckpt_capacity > 0");
        if (pool->pool && ((uintptr_t)pool->pool & 15) != 0)
            return fail(KDA_ERR_INVALID_ARG, "state_pool must be 16-byte aligned");
    } else if (desc->ckpt_stride > 0 && !ckpts && desc->ckpt_capacity > 0) {
        return fail(KDA_ERR_INVALID_ARG, "ckpts is NULL but ckpt_capacity > 0");
    }
    if (fused && fused->conv_w && desc->conv_width < 1)
        return fail(KDA_ERR_INVALID_ARG, "conv_w given but conv_width is %d (must be 1 to %d)", desc->conv_width,
                    kda::kConvTaps);
    if (fused && fused->gate && (fused->gate == q || fused->gate == k || fused->gate == v || fused->gate == out))
        return fail(KDA_ERR_INVALID_ARG, "gate aliases q, k, v or out");
    if (!workspace) return fail(KDA_ERR_WORKSPACE, "workspace is NULL");
    if (workspace_bytes < L.total)
        return fail(KDA_ERR_WORKSPACE, "workspace %zu bytes < required %zu", workspace_bytes, L.total);
    if (((uintptr_t)workspace & 255) != 0) return fail(KDA_ERR_WORKSPACE, "workspace not 256-byte aligned");
    if (out && (out == q || out == k || out == v))
        return fail(KDA_ERR_INVALID_ARG, "out aliases an input");
    if (kda::use_tc_path(desc->dtype, desc->head_dim_k, desc->chunk) &&
        ((((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)out) & 15) != 0 ||
         ((uintptr_t)g & (desc->scalar_gate ? 3 : 7)) != 0))
        return fail(KDA_ERR_INVALID_ARG,
                    "q, k, v and out must be 16-byte aligned and g 8-byte aligned (4 with scalar_gate)");

    char *ws = (char *)workspace;
    kda::PrefillArgs a;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.init_state = init_state;
    a.cu_seqlens = cu_seqlens; a.out = out; a.final_state = final_state;
    a.ckpts = desc->ckpt_stride > 0 ? ckpts : nullptr;
    a.N = desc->num_seqs; a.H = desc->num_heads; a.D = desc->head_dim_k; a.C = desc->chunk;
    a.T = T; a.ckpt_stride = desc->ckpt_stride; a.ckpt_capacity = desc->ckpt_capacity;
    a.dtype = desc->dtype; a.max_chunks = L.max_chunks;
    a.status = (kda::DevStatus *)(ws + L.status);
    a.tab.cu = (int32_t *)(ws + L.cu);
    a.tab.chunk_off = (int32_t *)(ws + L.chunk_off);
    a.tab.ckpt_off = (int32_t *)(ws + L.ckpt_off);
    a.handoff = ws + L.handoff;
    a.handoff_bytes = L.carry - L.handoff;
    a.carry = L.plan.nseg > 1 ? (float *)(ws + L.carry) : nullptr;
    a.plan = L.plan;
    a.seq_cap_chunks = L.plan.nseg > 1 ? L.plan.covered() : 0;
    a.scalar_gate = desc->scalar_gate != 0;
    a.wait_limit = desc->wait_limit ? desc->wait_limit : kda::kDefaultWaitLimit;
    a.init_slots = a.final_slots = a.ckpt_slots = nullptr;
    a.pool_slots = 0;
    if (pool) {   // every state lives in the pool; a NULL table means none of that kind
        a.init_state = pool->init_slots ? pool->pool : nullptr;
        a.final_state = pool->final_slots ? pool->pool : nullptr;
        a.ckpts = desc->ckpt_stride > 0 && pool->ckpt_slots ? pool->pool : nullptr;
        a.init_slots = pool->init_slots;
        a.final_slots = pool->final_slots;
        a.ckpt_slots = pool->ckpt_slots;
        a.pool_slots = pool->slots;
    }
    a.conv_w = fused ? fused->conv_w : nullptr;
    a.conv_width = a.conv_w ? desc->conv_width : 0;
    a.conv_silu = a.conv_w ? desc->conv_silu : 0;
    a.gate = fused ? fused->gate : nullptr;
    a.conv_in = a.conv_w && a.conv_width > 1 ? fused->conv_in : nullptr;
    a.conv_out = a.conv_w && a.conv_width > 1 ? fused->conv_out : nullptr;
    a.stream = (cudaStream_t)stream;
    {
        const bool tc = kda::use_tc_path(a.dtype, a.D, a.C);
        const size_t rec = tc ? kda::tc_handoff_bytes_per_chunk() : kda::simt_handoff_bytes_per_chunk(a.D, a.C);
        a.bounds.tokens = T - debug_clip_tokens();
        a.bounds.records = (int64_t)(a.handoff_bytes / rec);
        a.bounds.states = pool ? pool->slots : a.N;
        a.bounds.ckpts = pool ? pool->slots : a.ckpt_capacity;
    }

    cudaError_t e;
    if (kda::use_tc_path(a.dtype, a.D, a.C)) {
        e = use_graph ? kda::launch_prefill_tc_graph(a) : kda::enqueue_prefill_tc(a, a.stream);
        if (e != cudaSuccess)
            return fail(KDA_ERR_CUDA, "prefill kernels: %s %s", cudaGetErrorString(e), kda::launch_failure_detail());
        return debug_finish(KDA_OK, a.stream);
    }
    if ((e = cudaMemsetAsync(a.status, 0, sizeof(int32_t), a.stream)) != cudaSuccess) return cuda_fail(e, "status reset");
    if ((e = kda::launch_seq_table(a)) != cudaSuccess) return cuda_fail(e, "sequence table");
    if ((e = kda::launch_prefill_simt(a)) != cudaSuccess)
        return fail(KDA_ERR_CUDA, "prefill kernels: %s", cudaGetErrorString(e));
    if (a.conv_out && (e = kda::launch_conv_tail(a)) != cudaSuccess) return cuda_fail(e, "convolution state");
    return debug_finish(KDA_OK, a.stream);
}
}  // namespace kda

extern "C" {

kda_status kda_prefill(const void *q, const void *k, const void *v, const float *g,
                       const float *beta, const float *init_state, const int32_t *cu_seqlens,
                       void *out, float *final_state, float *ckpts,
                       const kda_prefill_desc *desc, void *workspace, size_t workspace_bytes,
                       kda_stream_t stream)
{
    NvtxRange r("kda_prefill");
    return kda::prefill_call(q, k, v, g, beta, init_state, cu_seqlens, out, final_state, ckpts, desc, workspace,
                             workspace_bytes, stream, true);
}

kda_status kda_prefill_fused(const void *q, const void *k, const void *v, const float *g,
                             const float *beta, const float *init_state, const int32_t *cu_seqlens,
                             void *out, float *final_state, float *ckpts, const float *conv_w,
                             const void *conv_state_in, void *conv_state_out, const void *gate,
                             const kda_prefill_desc *desc, void *workspace, size_t workspace_bytes,
                             kda_stream_t stream)
{
    NvtxRange r("kda_prefill_fused");
    if (!conv_w && (conv_state_in || conv_state_out))
        return fail(KDA_ERR_INVALID_ARG, "a convolution state is given without conv_w");
    const kda::FusedArgs fused{conv_w, gate, conv_state_in, conv_state_out};
    return kda::prefill_call(q, k, v, g, beta, init_state, cu_seqlens, out, final_state, ckpts, desc, workspace,
                             workspace_bytes, stream, true, nullptr, &fused);
}

kda_status kda_prefill_pooled(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, const int32_t *cu_seqlens, void *out,
                              float *state_pool, int64_t pool_slots, const int32_t *init_slots,
                              const int32_t *final_slots, const int32_t *ckpt_slots,
                              const kda_prefill_desc *desc, void *workspace, size_t workspace_bytes,
                              kda_stream_t stream)
{
    NvtxRange r("kda_prefill_pooled");
    const kda::PoolArgs pool{state_pool, pool_slots, init_slots, final_slots, ckpt_slots};
    return kda::prefill_call(q, k, v, g, beta, nullptr, cu_seqlens, out, nullptr, nullptr, desc, workspace,
                             workspace_bytes, stream, true, &pool);
}

kda_status kda_prefill_status(void *workspace, kda_stream_t stream)
{
    if (!workspace) return fail(KDA_ERR_WORKSPACE, "workspace is NULL");
    int32_t code = 0;
    cudaError_t e = cudaMemcpyAsync(&code, workspace, sizeof code, cudaMemcpyDeviceToHost,
                                    (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    e = cudaMemsetAsync(workspace, 0, sizeof(int32_t), (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
    if (code == KDA_OK) return KDA_OK;
    if (code == KDA_ERR_CKPT_OVERFLOW)
        return fail(KDA_ERR_CKPT_OVERFLOW, "more checkpoints due than ckpt_capacity; extra snapshots dropped");
    if (code == KDA_ERR_INVALID_ARG)
        return fail(KDA_ERR_INVALID_ARG,
                    "malformed cu_seqlens (must start at 0, be non-decreasing, end at T) "
                    "or a sequence longer than max_seq_len");
    if (code == KDA_ERR_TIMEOUT) return fail(KDA_ERR_TIMEOUT, "a bounded device-side wait gave up");
    return fail((kda_status)code, "device reported status %d", code);
}

namespace {
kda_status decode_common(const void *q, const void *k, const void *v, const float *g, const float *beta,
                         float *state, const int32_t *slots, int64_t pool, int32_t m,
                         const int32_t *commit, void *out, int32_t N, int32_t H, int32_t Dk, int32_t Dv,
                         kda_dtype dtype, int32_t *status, kda_stream_t stream)
{
    if (N < 0 || H < 0 || m < 0) return fail(KDA_ERR_INVALID_ARG, "N, m and H must be >= 0");
    if ((int64_t)N * m * H > INT32_MAX) return fail(KDA_ERR_UNSUPPORTED, "N*m*H too large");
    if (Dk != Dv) return fail(KDA_ERR_UNSUPPORTED, "Dk (%d) != Dv (%d)", Dk, Dv);
    if (Dk != 64 && Dk != 128) return fail(KDA_ERR_UNSUPPORTED, "head dim %d not in {64, 128}", Dk);
    if (dtype != KDA_DTYPE_BF16 && dtype != KDA_DTYPE_FP32)
        return fail(KDA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if ((size_t)N * H * m == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !state || !out)
        return fail(KDA_ERR_INVALID_ARG, "q, k, v, g, beta, state and out must be non-NULL");
    if (((uintptr_t)state & 15) != 0) return fail(KDA_ERR_INVALID_ARG, "state must be 16-byte aligned");
    if (out == q || out == k || out == v || out == (void *)state)
        return fail(KDA_ERR_INVALID_ARG, "out aliases an input");
    const kda::Bounds bd{(int64_t)N * m - debug_clip_tokens(), 0, slots ? pool : N, 0};
    cudaError_t e = kda::launch_decode(q, k, v, g, beta, state, out, N, H, Dk, dtype, slots, pool, m,
                                       commit, status, bd, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel");
    return debug_finish(KDA_OK, (cudaStream_t)stream);
}
}  // namespace

kda_status kda_decode(const void *q, const void *k, const void *v, const float *g,
                      const float *beta, float *state, void *out, int32_t N, int32_t H,
                      int32_t Dk, int32_t Dv, kda_dtype dtype, kda_stream_t stream)
{
    NvtxRange r("kda_decode");
    return decode_common(q, k, v, g, beta, state, nullptr, 0, 1, nullptr, out, N, H, Dk, Dv, dtype, nullptr,
                         stream);
}

kda_status kda_decode_fused(const void *q, const void *k, const void *v, const float *g,
                            const float *beta, float *state, void *conv_state, const float *conv_w,
                            const void *gate, void *out, int32_t N, int32_t H, int32_t Dk, int32_t Dv,
                            kda_dtype dtype, int32_t conv_width, int32_t conv_silu, kda_stream_t stream)
{
    NvtxRange r("kda_decode_fused");
    if (conv_w && (conv_width < 1 || conv_width > kda::kConvTaps))
        return fail(KDA_ERR_UNSUPPORTED, "conv_width %d not in [1, %d]", conv_width, kda::kConvTaps);
    if (conv_silu != 0 && conv_silu != 1) return fail(KDA_ERR_INVALID_ARG, "conv_silu must be 0 or 1");
    if (!conv_w && conv_state) return fail(KDA_ERR_INVALID_ARG, "conv_state given without conv_w");
    if (N < 0 || H < 0) return fail(KDA_ERR_INVALID_ARG, "N and H must be >= 0");
    if ((int64_t)N * H > INT32_MAX) return fail(KDA_ERR_UNSUPPORTED, "N*H too large");
    if (Dk != Dv) return fail(KDA_ERR_UNSUPPORTED, "Dk (%d) != Dv (%d)", Dk, Dv);
    if (Dk != 64 && Dk != 128) return fail(KDA_ERR_UNSUPPORTED, "head dim %d not in {64, 128}", Dk);
    if (dtype != KDA_DTYPE_BF16 && dtype != KDA_DTYPE_FP32)
        return fail(KDA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if ((size_t)N * H == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !state || !out)
        return fail(KDA_ERR_INVALID_ARG, "q, k, v, g, beta, state and out must be non-NULL");
    if (((uintptr_t)state & 15) != 0) return fail(KDA_ERR_INVALID_ARG, "state must be 16-byte aligned");
    if (out == q || out == k || out == v || out == (void *)state || (gate && out == gate))
        return fail(KDA_ERR_INVALID_ARG, "out aliases an input");
    const kda::DecodeFused f{conv_w, conv_w ? conv_width : 0, conv_silu, conv_w ? conv_state : nullptr, gate};
    const kda::Bounds bd{(int64_t)N - debug_clip_tokens(), 0, N, 0};
    cudaError_t e = kda::launch_decode_fused(q, k, v, g, beta, state, out, N, H, Dk, dtype, f, bd,
                                             (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel");
    return debug_finish(KDA_OK, (cudaStream_t)stream);
}

kda_status kda_decode_paged(const void *q, const void *k, const void *v, const float *g,
                            const float *beta, float *state_pool, int64_t pool_slots,
                            const int32_t *slot_ids, void *out, int32_t N, int32_t H, int32_t Dk,
                            int32_t Dv, kda_dtype dtype, int32_t *status, kda_stream_t stream)
{
    NvtxRange r("kda_decode_paged");
    if (pool_slots < 0) return fail(KDA_ERR_INVALID_ARG, "pool_slots must be >= 0");
    if (N > 0 && H > 0 && !slot_ids) return fail(KDA_ERR_INVALID_ARG, "slot_ids is NULL");
    return decode_common(q, k, v, g, beta, state_pool, slot_ids, pool_slots, 1, nullptr, out, N, H, Dk, Dv,
                         dtype, status, stream);
}

kda_status kda_decode_multi(const void *q, const void *k, const void *v, const float *g,
                            const float *beta, float *state, int64_t pool_slots, const int32_t *slot_ids,
                            const int32_t *commit_len, void *out, int32_t N, int32_t m, int32_t H,
                            int32_t Dk, int32_t Dv, kda_dtype dtype, int32_t *status, kda_stream_t stream)
{
    NvtxRange r("kda_decode_multi");
    if (slot_ids && pool_slots < 0) return fail(KDA_ERR_INVALID_ARG, "pool_slots must be >= 0");
    return decode_common(q, k, v, g, beta, state, slot_ids, slot_ids ? pool_slots : 0, m, commit_len, out,
                         N, H, Dk, Dv, dtype, slot_ids ? status : nullptr, stream);
}

}  // extern "C"
