// kda_common.cuh -- small device helpers shared by the KDA kernels of this
// library (element conversion, warp reductions, cache-hinted loads/stores),
// and the internal launcher interface between the C ABI and the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

// ---------------------------------------------------------------- elements
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ------------------------------------------------------------ workspace map
// Device status word values (a subset of kda_status, stored as int32).
struct DevStatus {
    int32_t code;        // 0 or a negative kda_status
    int32_t pad[63];
};

// Records `code` in the status word unless an earlier condition is already
// recorded there (the first one reported wins).
__device__ __forceinline__ void record_status(DevStatus *st, int32_t code)
{
    atomicCAS(&st->code, 0, code);
}

// ------------------------------------------------------------ debug build
// Compiled with -DKDA_DEBUG, the kernels check every global index they derive
// from data against the extent of its buffer before the access; an index
// outside it skips the access and the first one is recorded in a device word
// of its translation unit, which the entry point reads once the stream is
// synchronised.  Without KDA_DEBUG every check is the constant `true`.
struct Bounds {
    int64_t tokens;      // token rows of q, k, v, g, beta, out, gate (each row H x D)
    int64_t records;     // K1 -> K2 records (per chunk and head) the workspace holds
    int64_t states;      // [H, D, D] blocks of the initial / final states (N, or the pool's slots)
    int64_t ckpts;       // [H, D, D] checkpoint blocks (the capacity, or the pool's slots)
};
enum DbgSite : int32_t { kDbgTokenRow = 1, kDbgRecord = 2, kDbgState = 3, kDbgCkpt = 4 };
struct DbgWord {
    int32_t code;        // 0, or KDA_ERR_BOUNDS once a check failed
    int32_t site;        // DbgSite of the first failed check
    int64_t index, extent;
};
#ifdef KDA_DEBUG
constexpr bool kDebug = true;
static __device__ DbgWord g_dbg;
#else
constexpr bool kDebug = false;
#endif

// True when 0 <= i < n; otherwise (debug build) records the first such index.
__device__ __forceinline__ bool dbg_in(int64_t i, int64_t n, DbgSite site)
{
#ifdef KDA_DEBUG
    if (i >= 0 && i < n) return true;
    if (atomicCAS(&g_dbg.code, 0, (int32_t)KDA_ERR_BOUNDS) == 0) {
        g_dbg.site = site;
        g_dbg.index = i;
        g_dbg.extent = n;
    }
    return false;
#else
    (void)i; (void)n; (void)site;
    return true;
#endif
}

// Rows of a block of `rows` token rows from row t0 that lie inside the token
// buffers: `rows` itself, or (debug build) fewer, recording the first row past
// the end.
__device__ __forceinline__ int dbg_rows(int64_t t0, int rows, const Bounds &bd)
{
    if constexpr (kDebug) {
        if (rows > 0 && !dbg_in(t0 + rows - 1, bd.tokens, kDbgTokenRow)) {
            const int64_t r = bd.tokens - t0;
            return r < 0 ? 0 : (int)r;
        }
    }
    return rows;
}

// Defines `DbgWord name()`, which reads and clears this translation unit's
// device word (host side; the stream must be synchronised), or returns a
// cleared word without KDA_DEBUG.
#ifdef KDA_DEBUG
#define KDA_DBG_TAKE(name)                                                  \
    DbgWord name()                                                          \
    {                                                                       \
        DbgWord w{}, z{};                                                   \
        if (cudaMemcpyFromSymbol(&w, g_dbg, sizeof w) != cudaSuccess ||     \
            cudaMemcpyToSymbol(g_dbg, &z, sizeof z) != cudaSuccess)         \
            (void)cudaGetLastError();                                       \
        return w;                                                           \
    }
#else
#define KDA_DBG_TAKE(name) \
    DbgWord name() { return DbgWord{}; }
#endif
DbgWord dbg_take_prefill_tc();
DbgWord dbg_take_prefill_simt();
DbgWord dbg_take_decode();

// Largest magnitude of the exponent of one factor of the chunked form's
// decayed Gram product.  Per key channel the in-chunk log-decays b_r are
// referred to the midpoint B of their range (b_r - B and B - b_r), so the
// factors stay within e^{+-kMaxDecayExp} while the chunk's total decay stays
// below 2 * kMaxDecayExp; beyond that the factors are clamped (finite, no
// longer exact) and the chunk is reported as KDA_ERR_UNSUPPORTED.
constexpr float kMaxDecayExp = 80.f;

// Per-call table produced on the device from cu_seqlens (no host sync):
//   cu[n]        token offset of sequence n (a validated copy)
//   chunk_off[n] first global chunk index of sequence n (prefix sum of ceil(len/C))
//   ckpt_off[n]  first checkpoint slot of sequence n (prefix sum of floor(len/stride))
struct SeqTable {
    int32_t *cu;
    int32_t *chunk_off;
    int32_t *ckpt_off;
};

// ------------------------------------------------------------ launchers
// Segment plan of the tensor-core prefill.  Every sequence is cut into
// segments of G local chunks; the preparation kernel (K1) of segment s + 1
// runs on the caller's stream while the recurrence kernel (K2) of segment s
// runs on a side stream, and a segment's K1 -> K2 records occupy one of R ring
// slots of G chunks per sequence.  The state crosses a segment boundary
// through an fp32 carry buffer.  nseg == 1: one K1 and one K2 launch over
// compactly indexed records (no ring slots, no carry).
constexpr int kMaxSegments = 256;
struct SegPlan {
    int G;      // ring slot capacity: chunks per sequence of the longest segment
    int nseg;   // number of segments
    int R;      // ring slots
    int k2_ctas;   // CTAs of each recurrence launch (each runs chains one after another); 0: one per chain
    int lo[kMaxSegments + 1];   // segment s: local chunks [lo[s], lo[s + 1]) of every sequence
    int begin(int s) const { return lo[s]; }
    int count(int s) const { return lo[s + 1] - lo[s]; }
    int covered() const { return lo[nseg]; }
};

struct PrefillArgs {
    const void *q, *k, *v;
    const float *g, *beta, *init_state;
    const int32_t *cu_seqlens;   // may be NULL
    void *out;
    float *final_state, *ckpts;
    int N, H, D, C;
    int64_t T;
    int ckpt_stride;
    int64_t ckpt_capacity;
    kda_dtype dtype;
    int max_chunks;              // upper bound of chunks over all sequences
    DevStatus *status;
    SeqTable tab;
    void *handoff;               // K1 -> K2 buffer (the ring when plan.nseg > 1)
    size_t handoff_bytes;
    float *carry;                // [N, H, D, D] state between segments (plan.nseg > 1)
    SegPlan plan;
    int seq_cap_chunks;          // chunks any sequence may have (0 = unbounded)
    bool scalar_gate;            // g is [T, H] (one decay per head), else [T, H, Dk]
    uint32_t wait_limit;         // polls before a bounded device-side wait gives up
    // State pool (kda_prefill_pooled): init_state, final_state and ckpts then
    // all point to a pool of pool_slots [H, D, D] slots and these tables map
    // sequence n (or checkpoint j) to its slot; NULL tables: dense arrays.
    const int32_t *init_slots, *final_slots, *ckpt_slots;
    int64_t pool_slots;
    // Fused prologue / epilogue (kda_prefill_fused): short-convolution taps
    // [3, conv_width, H, D] (NULL: none) with optional SiLU, output gate [T, H, Dv]
    const float *conv_w;
    int conv_width, conv_silu;
    const void *gate;
    // convolution state [N, 3, conv_width - 1, H, D] (dtype of q): the rows before
    // each sequence (NULL: zeros) and, written at the end of the call, after it
    const void *conv_in;
    void *conv_out;
    Bounds bounds;               // extents the debug build checks indices against
    cudaStream_t stream;
};

// Where a prefill's recurrence reads initial states and writes final states
// and checkpoints: dense [N, H, D, D] / [capacity, H, D, D] arrays (NULL slot
// tables) or slots of one pool (kda_prefill_pooled).
struct StateIO {
    const float *init;           // NULL: zero initial states
    float *fin;                  // NULL: final states not written
    float *ckpts;                // NULL: no checkpoints
    const int32_t *init_slots, *final_slots, *ckpt_slots;
    int64_t pool;                // slots of the pool (with slot tables)
    int64_t capacity;            // checkpoint slots
    int stride;                  // checkpoint stride in tokens (0: none)
};

inline StateIO state_io(const PrefillArgs &a)
{
    return StateIO{a.init_state, a.final_state, a.ckpts, a.init_slots, a.final_slots, a.ckpt_slots,
                   a.pool_slots, a.ckpt_capacity, a.ckpts ? a.ckpt_stride : 0};
}

// Slot of entry i under an optional slot table: the table's entry when it is in
// [0, pool), -1 otherwise (no state there); without a table, i itself.
__device__ __forceinline__ int64_t pool_slot(const int32_t *slots, int64_t i, int64_t pool)
{
    if (!slots) return i;
    const int64_t s = slots[i];
    return (s >= 0 && s < pool) ? s : -1;
}

// Bytes of the K1 -> K2 handoff buffer for one (chunk, head).
size_t simt_handoff_bytes_per_chunk(int D, int C);

// Bytes of the tensor-core path's K1 -> K2 record for one (chunk, head).
size_t tc_handoff_bytes_per_chunk();

// The tensor-core path serves bf16 inputs with Dk = Dv = 128 and chunk 64;
// everything else runs on the fp32 CUDA-core path.
inline bool use_tc_path(kda_dtype dtype, int D, int C)
{
    return dtype == KDA_DTYPE_BF16 && D == 128 && C == 64;
}

// Segment plan of the tensor-core path for a validated descriptor.
SegPlan tc_segment_plan(const kda_prefill_desc *desc);

// Validates `desc` and returns the workspace bytes kda_prefill needs for it
// (on error: the status, with the thread-local message set).
kda_status prefill_workspace_bytes(const kda_prefill_desc *desc, size_t *bytes);
// A state pool and its slot tables (kda_prefill_pooled).
struct PoolArgs {
    float *pool;
    int64_t slots;
    const int32_t *init_slots, *final_slots, *ckpt_slots;
};
// The fused prologue / epilogue of kda_prefill_fused.
struct FusedArgs {
    const float *conv_w;
    const void *gate;
    const void *conv_in;
    void *conv_out;
};
// Taps of the short convolution as the kernels apply it (narrower
// convolutions are padded with zero taps on the older side).
constexpr int kConvTaps = 4;
// kda_prefill's body; use_graph = false launches every kernel directly (no
// CUDA graph is captured or instantiated: the no-allocation entry point).
// With `pool`, states and checkpoints live in pool slots (init_state,
// final_state and ckpts are ignored).
kda_status prefill_call(const void *q, const void *k, const void *v, const float *g, const float *beta,
                        const float *init_state, const int32_t *cu_seqlens, void *out, float *final_state,
                        float *ckpts, const kda_prefill_desc *desc, void *workspace, size_t workspace_bytes,
                        kda_stream_t stream, bool use_graph, const PoolArgs *pool = nullptr,
                        const FusedArgs *fused = nullptr);

// Default number of polls of a bounded device-side wait.
constexpr uint32_t kDefaultWaitLimit = 1u << 22;
// Sets the thread-local message that kda_last_error() returns; returns `s`.
kda_status fail_with_message(kda_status s, const char *fmt, ...);

cudaError_t launch_seq_table(const PrefillArgs &a);
// Writes the convolution state after each sequence (a.conv_out), last in a call.
cudaError_t launch_conv_tail(const PrefillArgs &a);
cudaError_t launch_prefill_simt(const PrefillArgs &a);
cudaError_t launch_prefill_tc(const PrefillArgs &a);
// The whole tensor-core call (status reset, sequence table, K1/K2 segments) on
// `stream`, and the same call replayed from a cached CUDA graph.
cudaError_t enqueue_prefill_tc(PrefillArgs a, cudaStream_t stream);
cudaError_t launch_prefill_tc_graph(const PrefillArgs &a);
// Kernel attributes noted by the last failed tensor-core launch on this thread ("" if none).
const char *launch_failure_detail();
// Streaming multiprocessors of the current device (cached per device).
int64_t device_sm_count();
cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, float *state, void *out, int N, int H, int D,
                          kda_dtype dtype, const int32_t *slots, int64_t pool, int m,
                          const int32_t *commit, int32_t *status, const Bounds &bd, cudaStream_t stream);
// The fused decode step (kda_decode_fused): convolution with a per-sequence
// history, the step, the output gate.
struct DecodeFused {
    const float *conv_w;   // [3, W, H, D] or NULL
    int conv_width, conv_silu;
    void *conv_state;      // [N, 3, W - 1, H, D] dtype, read and advanced (NULL: zeros, not kept)
    const void *gate;      // [N, H, D] dtype or NULL
};
cudaError_t launch_decode_fused(const void *q, const void *k, const void *v, const float *g,
                                const float *beta, float *state, void *out, int N, int H, int D,
                                kda_dtype dtype, const DecodeFused &f, const Bounds &bd, cudaStream_t stream);

}  // namespace kda
