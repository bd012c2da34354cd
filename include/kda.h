/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention core library.
 *
 * The library computes, per sequence and head, the KDA recurrence that the
 * page "Kimi K3 reconstructs long-context inference efficiency through KDA,
 * cross-depth attention, and latent expert routing" describes in its section
 * "Methodology notes" (Delta Rule, per-channel diagonal decay, L2-normalised
 * q/k) and its section "Key data" (cost figures):
 *
 *     qh = q / sqrt(|q|^2 + 1e-6),   kh = k / sqrt(|k|^2 + 1e-6)    (fp32)
 *     S' = Diag(exp g_t) S_{t-1}                      key rows decay
 *     S_t = S' + beta_t kh (v_t - S'^T kh)^T          delta-rule step
 *     o_t = S_t^T qh                                  reads the updated state
 *
 * with S an fp32 Dk x Dv state per (sequence, head).
 *
 * Conventions shared by every entry point
 *   - All pointers are DEVICE pointers into contiguous, row-major buffers
 *     that the caller owns and allocates (the library allocates no buffer;
 *     the tensor-core prefill creates, once per host thread and device, a
 *     side stream, a few events and a capture stream, and keeps up to 8
 *     executable CUDA graphs, one per launch structure (number of
 *     segments): each kda_prefill call is captured on that stream and
 *     replayed from the graph of its structure, its launch parameters
 *     updated in place, which shortens the gaps between its kernels; inside
 *     a caller's own stream capture, and in kda_prefill_noalloc, the kernels
 *     are launched directly).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  No entry point synchronises the stream.  Tensor-core prefill
 *     calls made from one host thread replay the same cached CUDA graphs, so
 *     the GPU runs them one after another even when they are enqueued on
 *     different streams; calls from different threads do not share graphs.
 *     The per-thread side stream, events and graphs live until the process
 *     exits.
 *   - g <= 0 (alpha = exp(g) is a decay); see kda_prefill for the range.
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid call returns a negative kda_status and touches no buffer.
 *     kda_last_error() then returns a message (thread-local).
 *   - Conditions only the device can see (malformed cu_seqlens, checkpoint
 *     capacity too small) are recorded in a status word inside the caller's
 *     workspace; kda_prefill_status() reads it back (this one call
 *     synchronises the stream).
 *   - Supported shapes: Dk == Dv in {64, 128}; chunk == 64; dtype of q, k, v
 *     and out bf16 or fp32; g, beta, states and checkpoints always fp32.
 *
 * Debug build (libkda_debug.so: the same sources compiled with -DKDA_DEBUG,
 * the same symbols and results)
 *   - Every global index that the kernels derive from data (token rows from
 *     cu_seqlens, records in the workspace, state, pool-slot and checkpoint
 *     blocks) is checked against the extent of its buffer before the access.
 *     An index outside it skips the access (no trap, nothing outside the
 *     buffer is touched; the results are then undefined) and the first such
 *     index is recorded in a device word.
 *   - Every entry point that launched work then synchronises `stream` (not
 *     while the stream is being captured) and returns KDA_ERR_BOUNDS if a
 *     check failed, with kda_last_error() naming the buffer, the index and
 *     the extent (device conditions of the release build, such as those
 *     kda_prefill_status reports, are reported as there).
 *   - Environment variable KDA_DEBUG_CLIP_TOKENS=n (debug build only): the
 *     checks take the token-row buffers of every call (q, k, v, g, beta, out,
 *     gate) to be n rows shorter than the call's size says, so that a test can
 *     make the last rows fail the check while the memory behind them exists.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (the same type as cudaStream_t / CUstream). */
typedef struct CUstream_st *kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = -1,    /* null pointer, bad size, malformed cu_seqlens */
    KDA_ERR_UNSUPPORTED = -2,    /* valid but not implemented (head dim, chunk) */
    KDA_ERR_CUDA = -3,           /* a CUDA launch or runtime call failed */
    KDA_ERR_CKPT_OVERFLOW = -4,  /* more checkpoints due than ckpt_capacity slots */
    KDA_ERR_WORKSPACE = -5,      /* workspace missing or smaller than required */
    KDA_ERR_TIMEOUT = -6,        /* a bounded device-side wait gave up */
    KDA_ERR_BOUNDS = -7          /* debug build: a global index outside its buffer (access skipped) */
} kda_status;

typedef enum {
    KDA_DTYPE_BF16 = 0,          /* q, k, v, out are bf16 */
    KDA_DTYPE_FP32 = 1           /* q, k, v, out are fp32 */
} kda_dtype;

/*
 * Shape and options of one prefill call.
 *   num_seqs       N >= 1.
 *   total_tokens   T >= 0: rows of q/k/v/g/beta/out.  With cu_seqlens == NULL
 *                  the batch is N equal-length sequences laid out one after
 *                  another (T must be a multiple of N).
 *   num_heads      H >= 1.
 *   head_dim_k/v   Dk, Dv (must be equal, 64 or 128).
 *   dtype          element type of q, k, v and out.
 *   chunk          C, the block length of the chunked form (64).
 *   ckpt_stride    0 = no checkpoints; else a multiple of chunk: after every
 *                  ckpt_stride tokens of a sequence the state is copied to
 *                  the next checkpoint slot (the page's prefix-cache
 *                  snapshots every 32K tokens, zsxq post on SemiAnalysis'
 *                  Kimi K3 analysis, section "五、KV缓存效率与服务性能").
 *   ckpt_capacity  number of [H, Dk, Dv] slots in `ckpts`.
 *   max_seq_len    an upper bound on the length of every sequence, or 0 when
 *                  unknown (total_tokens is assumed).  The tensor-core path
 *                  (bf16, Dk = Dv = 128) may split every sequence into
 *                  segments of `segment_chunks` chunks and run the
 *                  preparation of segment s + 1 concurrently with the
 *                  recurrence over segment s; max_seq_len bounds the number
 *                  of segments and so the workspace.  A sequence longer than
 *                  the bound is reported as KDA_ERR_INVALID_ARG by
 *                  kda_prefill_status and its tail is not computed.
 *   segment_chunks 0 = chosen by the library (from num_seqs x num_heads and
 *                  the sequence bound); otherwise the number of chunks per
 *                  sequence in one segment, raised where needed so that
 *                  there are at most 256 segments.  A tuning knob only: the
 *                  results are bit-identical for every value, since the
 *                  state crosses a segment boundary in fp32 unchanged.
 *   scalar_gate    0: g is [T, H, Dk], one log-decay per key channel (KDA).
 *                  1: g is [T, H], one log-decay per token and head applied
 *                  to every key channel (the scalar-gate Gated DeltaNet the
 *                  zsxq post on SemiAnalysis' Kimi K3 analysis, section
 *                  "一、Kimi Delta Attention（KDA）", contrasts KDA with);
 *                  the results equal those of the per-channel form with
 *                  the gate repeated over the channels.
 *   recurrence_ctas 0 = chosen by the library.  Otherwise, when the
 *                  tensor-core path splits the call into segments, the number
 *                  of CTAs of each recurrence launch (each runs its share of
 *                  the sequence x head chains one after another); the rest of
 *                  the GPU prepares the next segment meanwhile.  A tuning knob
 *                  only: results are bit-identical for every value.
 *   conv_width     taps of the short convolution of kda_prefill_fused (1 to
 *                  4; 0 when there is none).  Ignored by the other entry points.
 *   conv_silu      1: the convolution's output passes through x*sigmoid(x)
 *                  (kda_prefill_fused only); 0: no activation.
 *   wait_limit     0 = default.  Otherwise the number of polls after which a
 *                  wait of the tensor-core kernels on an asynchronous step
 *                  (a copy, a tensor-core product, another role of the same
 *                  CTA) gives up: the kernel then drains its own work in
 *                  flight, records KDA_ERR_TIMEOUT and returns, and the
 *                  call's results are undefined.  A diagnostic: small values
 *                  exercise that path; the default (2^22 polls) is far above
 *                  any wait a correct call makes.
 */
typedef struct {
    int32_t num_seqs;
    int64_t total_tokens;
    int32_t num_heads;
    int32_t head_dim_k;
    int32_t head_dim_v;
    kda_dtype dtype;
    int32_t chunk;
    int32_t ckpt_stride;
    int64_t ckpt_capacity;
    int64_t max_seq_len;
    int32_t segment_chunks;
    int32_t scalar_gate;
    int32_t recurrence_ctas;
    int32_t conv_width;
    int32_t conv_silu;
    uint32_t wait_limit;
} kda_prefill_desc;

/*
 * Bytes of device workspace kda_prefill needs for `desc` (0 if desc is
 * invalid).  The workspace is caller-owned scratch; it holds the per-chunk
 * table, the device status word and the handoff between the preparation and
 * recurrence kernels.  One workspace must not be shared by calls that can run
 * concurrently.
 */
size_t kda_prefill_workspace_size(const kda_prefill_desc *desc);

/*
 * Number of kernel launches one kda_prefill call with this descriptor
 * enqueues (a sequence table, then one preparation and one recurrence launch
 * per segment), or -1 for an invalid descriptor (kda_last_error() says why).
 * Host-only: touches no device state.
 */
int32_t kda_prefill_launch_count(const kda_prefill_desc *desc);

/*
 * Chunked prefill over packed sequences (K1 tensor preparation + K2 blockwise
 * recurrence; page "Kimi K3 reconstructs long-context inference efficiency
 * ...", section "Methodology notes", item "System optimization: FlashKDA";
 * zsxq post, section "一、Kimi Delta Attention（KDA）": chunk-level
 * parallelism through the UT transform).
 *
 *   q, k        [T, H, Dk]  dtype          (normalised inside, in fp32)
 *   v           [T, H, Dv]  dtype
 *               The tensor-core path (bf16, Dk = Dv = 128) takes q, k, v and
 *               the state as f16 tensor-core operands: every q and k row
 *               needs an L2 norm below 65504, every v and state entry a
 *               magnitude below 65504.  The debug build reports a q, k or v
 *               beyond this as KDA_ERR_UNSUPPORTED (kda_prefill_status);
 *               the release build does not check it.
 *   g           [T, H, Dk]  fp32  log-decay, alpha = exp(g) ([T, H] when
 *                                 desc->scalar_gate), g <= 0.  Per key
 *                                 channel, the decay of one chunk of 64
 *                                 tokens (-sum g) must stay below 160; a
 *                                 chunk beyond it is computed with clamped
 *                                 decay factors (finite, inexact) and
 *                                 reported as KDA_ERR_UNSUPPORTED
 *   beta        [T, H]      fp32
 *   init_state  [N, H, Dk, Dv] fp32, or NULL for zeros
 *   cu_seqlens  [N + 1] int32 token offsets (0 = cu[0] <= ... <= cu[N] = T),
 *               or NULL for N equal-length sequences
 *   out         [T, H, Dv]  dtype          (written)
 *   final_state [N, H, Dk, Dv] fp32 or NULL; may alias init_state
 *   ckpts       [ckpt_capacity, H, Dk, Dv] fp32, or NULL when ckpt_stride == 0;
 *               slots are filled in sequence order, then snapshot order; a
 *               sequence of length L emits floor(L / ckpt_stride) snapshots
 *   workspace   >= kda_prefill_workspace_size(desc) bytes, 256-byte aligned
 *
 * out must not alias any input.  Returns KDA_OK once the work is enqueued.
 */
kda_status kda_prefill(const void *q, const void *k, const void *v, const float *g,
                       const float *beta, const float *init_state, const int32_t *cu_seqlens,
                       void *out, float *final_state, float *ckpts,
                       const kda_prefill_desc *desc, void *workspace, size_t workspace_bytes,
                       kda_stream_t stream);

/*
 * Reads (and clears) the device status word of `workspace` after the work
 * queued on `stream`: KDA_OK, KDA_ERR_INVALID_ARG (malformed cu_seqlens, or a
 * sequence longer than max_seq_len; the affected sequences were skipped),
 * KDA_ERR_CKPT_OVERFLOW (snapshots beyond ckpt_capacity were dropped),
 * KDA_ERR_UNSUPPORTED (a chunk's decay exceeded the range stated for g; in
 * the debug build also q, k or v beyond the f16 range stated for them) or
 * KDA_ERR_TIMEOUT (a bounded device-side wait gave up).  The first condition
 * recorded during the call is the one reported.  Synchronises `stream`.
 */
kda_status kda_prefill_status(void *workspace, kda_stream_t stream);

/*
 * One decode step for N sequences x H heads, state updated in place (page
 * "Kimi K3 reconstructs long-context inference efficiency ...", section "Key
 * data": about 7*D^2 FLOPs and 8*D^2 bytes of fp32 state traffic per head).
 *
 *   q, k   [N, H, Dk] dtype;   v [N, H, Dv] dtype;   g [N, H, Dk] fp32;
 *   beta   [N, H] fp32;        state [N, H, Dk, Dv] fp32, read and written;
 *   out    [N, H, Dv] dtype    (written; must not alias the inputs or state)
 */
kda_status kda_decode(const void *q, const void *k, const void *v, const float *g,
                      const float *beta, float *state, void *out, int32_t N, int32_t H,
                      int32_t Dk, int32_t Dv, kda_dtype dtype, kda_stream_t stream);

/*
 * kda_prefill without a workspace argument, for callers that cannot allocate
 * device memory (a framework that owns every allocation, a runtime that
 * forbids cudaMalloc after start-up).  The KDA pages have no counterpart of
 * this entry point; it exists only for such callers.
 *
 * Arguments are those of kda_prefill minus the workspace.  The scratch is a
 * fixed device array of KDA_NOALLOC_SCRATCH_BYTES built into the library:
 * every GPU that loads the library keeps it resident until the process exits.
 * When the automatic plan (desc->segment_chunks 0) of the tensor-core path
 * needs more than the array, the call takes the longest segments that fit:
 * one segment if every record fits, else the largest segment_chunks whose
 * ring and carry fit (the results are the same for every segment length).
 * A call that fits no plan returns KDA_ERR_UNSUPPORTED before any work is
 * queued, as does one with an explicit segment_chunks whose
 * kda_prefill_workspace_size() exceeds the array.  The need is about 90.6 KB
 * per chunk of 64 tokens and head for the bf16 path with Dk = Dv = 128 in
 * one segment (so about 360 chunk-heads, e.g. 11 chunks of 32 heads); a
 * smaller desc->segment_chunks bounds it by two ring slots of that many
 * chunks of every sequence and head plus 64 KB of fp32 carry per sequence
 * and head (segment_chunks = 1 with 32 heads: about 6 MB plus 2 MB per
 * sequence).  Nothing is allocated: no
 * cudaMalloc, cudaFree or allocating library routine is called.
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it; make that first call before any stream
 * capture begins.  All calls share the one array, which keeps the previous
 * call's contents; the parts that must start at zero are cleared by each
 * call.  Calls that can overlap on the GPU race on the array and must be
 * ordered by the caller.  Device-detected conditions (malformed cu_seqlens,
 * too few checkpoint slots) are not reported by this entry point: use
 * kda_prefill and kda_prefill_status when they matter.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
kda_status kda_prefill_noalloc(const void *q, const void *k, const void *v, const float *g,
                               const float *beta, const float *init_state,
                               const int32_t *cu_seqlens, void *out, float *final_state,
                               float *ckpts, const kda_prefill_desc *desc, kda_stream_t stream);

/*
 * kda_prefill with the steps on either side of the recurrence fused into its
 * kernels (page "Kimi K3 reconstructs long-context inference efficiency
 * ...", section "Methodology notes", item "Memory control: Kimi Delta
 * Attention": KDA combines a short convolution, the L2 normalisation of q and
 * k, and an output forget gate with the recurrence):
 *   conv_w  [3, desc->conv_width, H, D] fp32, or NULL for no convolution: the
 *           taps for q, k and v of a causal depthwise convolution along the
 *           tokens of each sequence,
 *               x'[t] = sum_{i < W} conv_w[., i] * x[t - (W - 1) + i],
 *           with tokens before the sequence's first counted as zero (tap
 *           W - 1 multiplies the current token), then x' * sigmoid(x') when
 *           desc->conv_silu.  The preparation kernel convolves q, k and v as
 *           it loads them (the tensor-core path rounds the results to f16,
 *           11 significant bits, within the f16 range it requires of q, k
 *           and v; the fp32 path keeps fp32); the L2
 *           normalisation of q and k follows as in kda_prefill.
 *   conv_state_in   [N, 3, conv_width - 1, H, D] dtype of q, or NULL: the
 *           raw q, k, v rows before each sequence (oldest first), the tokens
 *           a prefill resumed mid-sequence (or a decode) would otherwise not
 *           see; NULL counts them as zeros.
 *   conv_state_out  same shape, or NULL: written, last, with the raw rows
 *           ending each sequence (reaching into conv_state_in for sequences
 *           shorter than conv_width - 1), the history kda_decode_fused or a
 *           later prefill continues from; may be conv_state_in itself.
 *   gate    [T, H, Dv] dtype of out, or NULL for no gate: the output is
 *           o * sigmoid(gate), applied as the recurrence kernel stores it.
 * Every other argument, and the results without conv_w and gate, as
 * kda_prefill (with conv_state_out one launch more than
 * kda_prefill_launch_count reports).
 */
kda_status kda_prefill_fused(const void *q, const void *k, const void *v, const float *g,
                             const float *beta, const float *init_state, const int32_t *cu_seqlens,
                             void *out, float *final_state, float *ckpts, const float *conv_w,
                             const void *conv_state_in, void *conv_state_out, const void *gate,
                             const kda_prefill_desc *desc, void *workspace, size_t workspace_bytes,
                             kda_stream_t stream);

/*
 * kda_decode with the steps around the recurrence (the decode side of
 * kda_prefill_fused): each sequence's new q, k, v ([N, H, D] dtype) are
 * convolved with its history conv_state [N, 3, conv_width - 1, H, D] (dtype;
 * NULL: zeros), which the call then advances by the new raw rows; the step
 * runs as kda_decode on the dense states [N, H, Dk, Dv]; the output is
 * o * sigmoid(gate) (gate [N, H, Dv] dtype, or NULL).  conv_w [3, conv_width,
 * H, D] fp32 as for kda_prefill_fused, or NULL with conv_width 0 for no
 * convolution; conv_silu 0 or 1.
 */
kda_status kda_decode_fused(const void *q, const void *k, const void *v, const float *g,
                            const float *beta, float *state, void *conv_state, const float *conv_w,
                            const void *gate, void *out, int32_t N, int32_t H, int32_t Dk, int32_t Dv,
                            kda_dtype dtype, int32_t conv_width, int32_t conv_silu, kda_stream_t stream);

/*
 * Chunked prefill whose states live in a pool of slots (the prefill side of
 * a serving loop's state pool; the zsxq post on SemiAnalysis' Kimi K3
 * analysis, section "五、KV缓存效率与服务性能": the recurrent state is saved
 * every 32K tokens and at prompt boundaries, and a prefill resumes from such
 * a snapshot).  state_pool is [pool_slots, H, Dk, Dv] fp32; the slot tables
 * are int32 on the device:
 *   init_slots  [N]  sequence n starts from slot init_slots[n]; NULL, or a
 *                    slot outside [0, pool_slots), starts from zeros
 *   final_slots [N]  sequence n's final state is written to slot
 *                    final_slots[n]; NULL, or a slot out of range, skips it
 *   ckpt_slots  [ckpt_capacity]  snapshot j (numbered as kda_prefill's
 *                    checkpoint slots: sequence order, then snapshot order)
 *                    is written to slot ckpt_slots[j]; a slot out of range
 *                    skips it; required when ckpt_stride > 0 and
 *                    ckpt_capacity > 0
 * A sequence may end in the slot it started from (each reads its initial
 * state before writing its final state); otherwise the slots written by one
 * call must be distinct from each other and from every other sequence's
 * initial slot.  Everything else as kda_prefill, whose results this call
 * reproduces bit for bit on the gathered states.
 */
kda_status kda_prefill_pooled(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, const int32_t *cu_seqlens, void *out,
                              float *state_pool, int64_t pool_slots, const int32_t *init_slots,
                              const int32_t *final_slots, const int32_t *ckpt_slots,
                              const kda_prefill_desc *desc, void *workspace, size_t workspace_bytes,
                              kda_stream_t stream);

/*
 * kda_decode over a pool of states: the state of sequence n is slot
 * slot_ids[n] of state_pool [pool_slots, H, Dk, Dv] fp32 (updated in place),
 * so that a serving loop keeps sequences in fixed slots while its batch
 * changes (continuous batching; a prefill can write a sequence's slot as its
 * final_state, or resume from a checkpoint copied into a slot).  slot_ids is
 * int32 [N] on the device; a slot outside [0, pool_slots) marks a padding
 * row: its state is not touched and its output row is zero.  Slots of one call
 * must be distinct.  status: NULL, or a device int32 that the call sets to
 * KDA_ERR_INVALID_ARG (if it holds 0) when two sequences name the same valid
 * slot; their results are then undefined.  Everything else as kda_decode.
 */
kda_status kda_decode_paged(const void *q, const void *k, const void *v, const float *g,
                            const float *beta, float *state_pool, int64_t pool_slots,
                            const int32_t *slot_ids, void *out, int32_t N, int32_t H, int32_t Dk,
                            int32_t Dv, kda_dtype dtype, int32_t *status, kda_stream_t stream);

/*
 * Multi-token decode (a speculative-decoding verify step): each sequence runs
 * m tokens through the recurrence one after another with its state kept on
 * chip.  q, k, g: [N, m, H, Dk]; v, out: [N, m, H, Dv]; beta: [N, m, H].  The
 * state is dense [N, H, Dk, Dv] (slot_ids NULL, pool_slots ignored) or slot
 * slot_ids[n] of a pool as in kda_decode_paged.  commit_len (int32 [N] on the
 * device, or NULL for m) says after how many of its tokens each sequence's
 * state is written back (0 = not at all): a verify call computes the outputs
 * of all drafted tokens and commits the accepted prefix of the previous
 * step's drafts, or commits nothing and a second call commits the accepted
 * tokens.  Outputs of every token are written.  m = 1 with commit_len NULL is
 * kda_decode (kda_decode_paged with slots).  status as in kda_decode_paged
 * (checked only with slot_ids).
 */
kda_status kda_decode_multi(const void *q, const void *k, const void *v, const float *g,
                            const float *beta, float *state, int64_t pool_slots, const int32_t *slot_ids,
                            const int32_t *commit_len, void *out, int32_t N, int32_t m, int32_t H,
                            int32_t Dk, int32_t Dv, kda_dtype dtype, int32_t *status,
                            kda_stream_t stream);

/* Message for the last non-OK status returned on this thread ("" if none). */
const char *kda_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
