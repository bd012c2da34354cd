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
    cudaStream_t stream;
};

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
// kda_prefill's body; use_graph = false launches every kernel directly (no
// CUDA graph is captured or instantiated: the no-allocation entry point)
kda_status prefill_call(const void *q, const void *k, const void *v, const float *g, const float *beta,
                        const float *init_state, const int32_t *cu_seqlens, void *out, float *final_state,
                        float *ckpts, const kda_prefill_desc *desc, void *workspace, size_t workspace_bytes,
                        kda_stream_t stream, bool use_graph);
// Sets the thread-local message that kda_last_error() returns; returns `s`.
kda_status fail_with_message(kda_status s, const char *fmt, ...);

cudaError_t launch_seq_table(const PrefillArgs &a);
cudaError_t launch_prefill_simt(const PrefillArgs &a);
cudaError_t launch_prefill_tc(const PrefillArgs &a);
// The whole tensor-core call (status reset, sequence table, K1/K2 segments) on
// `stream`, and the same call replayed from a cached CUDA graph.
cudaError_t enqueue_prefill_tc(PrefillArgs a, cudaStream_t stream);
cudaError_t launch_prefill_tc_graph(const PrefillArgs &a);
// Kernel attributes noted by the last failed tensor-core launch on this thread ("" if none).
const char *launch_failure_detail();
cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, float *state, void *out, int N, int H, int D,
                          kda_dtype dtype, const int32_t *slots, int64_t pool, int m,
                          const int32_t *commit, cudaStream_t stream);

}  // namespace kda
