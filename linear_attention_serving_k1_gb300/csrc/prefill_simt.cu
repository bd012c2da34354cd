// prefill_simt.cu -- chunked KDA prefill on CUDA cores in fp32.
//
// The chunked form of the page "Kimi K3 reconstructs long-context inference
// efficiency through KDA, cross-depth attention, and latent expert routing"
// (section "Methodology notes", item "System optimization: FlashKDA": K1
// prepares decayed queries/keys, inverse transforms and causal matrices in
// parallel over chunks; K2 computes pseudo-values, outputs and updated states
// serially), with the UT transform of the zsxq post on SemiAnalysis' Kimi K3
// analysis (section "一、Kimi Delta Attention（KDA）").
//
// This is the all-fp32 path: every product is an fp32 FMA on CUDA cores and
// the K1 -> K2 handoff is kept in fp32, so it serves the fp32 workloads and
// head dims/dtypes the tensor-core path does not take.
//
// Per chunk (rows r < L valid, C = 64) with start state S0:
//   K1  qh, kh (fp32 L2 norm); b = inclusive cumsum of g; gamma = exp(b)
//       Qg = qh*gamma, Kg = kh*gamma, Kd = kh*exp(-b), Ke = Kd*gamma_last
//       Lm = strict-lower(diag(beta) Kg Kd^T); Tm = (I + Lm)^-1
//       Wk = Tm diag(beta) Kg, Uv = Tm diag(beta) V, M = incl-lower(Qg Kd^T)
//   K2  W = Uv - Wk S0; O = Qg S0 + M W; S1 = Diag(gamma_last) S0 + Ke^T W
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kC = 64;
constexpr int kThreads = 256;

// ---------------------------------------------------------------- seq table
// One CTA.  Validates cu_seqlens (or synthesises equal lengths), and writes the
// chunk and checkpoint prefix sums.  Serial over sequences on one thread: the
// number of sequences per call is small next to the token work.
__global__ void seq_table_kernel(const int32_t *__restrict__ cu_in, int N, int64_t T, int C,
                                 int stride, int64_t capacity, int cap_chunks, SeqTable tab,
                                 DevStatus *st)
{
    if (threadIdx.x != 0) return;
    bool ok = true, too_long = false;
    if (cu_in) {
        if (cu_in[0] != 0 || (int64_t)cu_in[N] != T) ok = false;
        for (int n = 0; n < N && ok; ++n)
            if (cu_in[n + 1] < cu_in[n]) ok = false;
    }
    int32_t chunks = 0, ck = 0;
    for (int n = 0; n <= N; ++n) {
        int32_t c0 = cu_in ? cu_in[n] : (int32_t)((T / N) * n);
        if (!ok) c0 = 0;
        tab.cu[n] = c0;
        tab.chunk_off[n] = chunks;
        tab.ckpt_off[n] = ck;
        if (n < N && ok) {
            int32_t c1 = cu_in ? cu_in[n + 1] : (int32_t)((T / N) * (n + 1));
            int32_t len = c1 - c0;
            chunks += (len + C - 1) / C;
            if (stride > 0) ck += len / stride;
            if (cap_chunks > 0 && (len + C - 1) / C > cap_chunks) too_long = true;
        }
    }
    if (!ok || too_long) st->code = (int32_t)KDA_ERR_INVALID_ARG;
    else if (stride > 0 && (int64_t)ck > capacity) st->code = (int32_t)KDA_ERR_CKPT_OVERFLOW;
}

// Sequence that owns global chunk gc (largest n with chunk_off[n] <= gc).
__device__ __forceinline__ int find_seq(const int32_t *chunk_off, int N, int gc)
{
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (chunk_off[mid] <= gc) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Handoff record of one (chunk, head), fp32:  Qg[C][D] Wk[C][D] Uv[C][D]
// Ke[C][D] M[C][C] gl[D].
struct Handoff {
    float *Qg, *Wk, *Uv, *Ke, *M, *gl;
};
__host__ __device__ __forceinline__ size_t handoff_floats(int D) {
    return (size_t)4 * kC * D + (size_t)kC * kC + D;
}
__device__ __forceinline__ Handoff handoff_at(float *base, size_t rec, int D)
{
    float *p = base + rec * handoff_floats(D);
    Handoff h;
    h.Qg = p; p += kC * D;
    h.Wk = p; p += kC * D;
    h.Uv = p; p += kC * D;
    h.Ke = p; p += kC * D;
    h.M = p; p += kC * kC;
    h.gl = p;
    return h;
}

// ---------------------------------------------------------------- K1
template <int D, typename T>
__global__ void __launch_bounds__(kThreads)
k1_simt_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
               const float *__restrict__ g, const float *__restrict__ beta, int N, int H,
               SeqTable tab, float *__restrict__ handoff, int scalar_gate, DevStatus *st,
               const float *__restrict__ conv_w, int conv_width, int conv_silu, const T *__restrict__ conv_in,
               Bounds bd)
{
    constexpr int P = D + 1;   // padded row pitch (bank-conflict free columns)
    extern __shared__ float smem[];
    float *Qg = smem;                 // [C][P]
    float *Kg = Qg + kC * P;          // [C][P]
    float *Kd = Kg + kC * P;          // [C][P]
    float *Vs = Kd + kC * P;          // [C][P]
    float *Lm = Vs + kC * P;          // [C][C+1]
    float *Tm = Lm + kC * (kC + 1);   // [C][C+1]
    float *bs = Tm + kC * (kC + 1);   // [C] beta
    float *mu = bs + kC;              // [D] e^B, B = half the chunk's log-decay per channel

    const int gc = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    if (gc >= tab.chunk_off[N]) return;
    const int n = find_seq(tab.chunk_off, N, gc);
    const int seq_t0 = tab.cu[n];
    const int t0 = tab.cu[n] + (gc - tab.chunk_off[n]) * kC;
    // (debug build: rows past the token buffers' end count as rows past the
    // sequence's end, and a record outside the workspace is not written)
    const int L = dbg_rows(t0, min(kC, tab.cu[n + 1] - t0), bd);
    if (!dbg_in((int64_t)gc * H + h, bd.records, kDbgRecord)) return;
    Handoff ho = handoff_at(handoff, (size_t)gc * H + h, D);

    // 1. rows: qh, kh (normalised, one warp per row), v, beta.  Rows >= L are zero.
    //    With conv_w (the fused prologue) q, k, v are first convolved along the
    //    sequence's tokens: x'[t] = sum_i w[i] x[t - (W - 1) + i] (tokens before the
    //    sequence's first count as zero), optionally x' sigmoid(x'), in fp32.
    const int warp = tid >> 5, lane = tid & 31;
    auto input = [&](const T *x, int t, int r, int d) -> float {   // x'[t0 + r] at channel d (or x itself)
        if (!conv_w) return to_f32(x[((size_t)(t0 + r) * H + h) * D + d]);
        float acc = 0.f;
        for (int i = 0; i < conv_width; ++i) {
            const int tau = t0 + r - (conv_width - 1) + i;
            const float wi = conv_w[(((size_t)t * conv_width + i) * H + h) * D + d];
            if (tau >= seq_t0)
                acc += wi * to_f32(x[((size_t)tau * H + h) * D + d]);
            else if (conv_in)   // the history before the sequence (oldest first)
                acc += wi * to_f32(conv_in[((((size_t)n * 3 + t) * (conv_width - 1) + (conv_width - 1 + tau - seq_t0)) * H + h) * D + d]);
        }
        return conv_silu ? acc / (1.f + expf(-acc)) : acc;
    };
    for (int r = warp; r < kC; r += kThreads / 32) {
        float qa[D / 32], ka[D / 32];
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int j = 0; j < D / 32; ++j) {
            const int d = lane + 32 * j;
            qa[j] = r < L ? input(q, 0, r, d) : 0.f;
            ka[j] = r < L ? input(k, 1, r, d) : 0.f;
            Vs[r * P + d] = r < L ? input(v, 2, r, d) : 0.f;
            sq += qa[j] * qa[j];
            sk += ka[j] * ka[j];
        }
        sq = rsqrtf(warp_sum(sq) + 1e-6f);
        sk = rsqrtf(warp_sum(sk) + 1e-6f);
#pragma unroll
        for (int j = 0; j < D / 32; ++j) {
            Qg[r * P + lane + 32 * j] = qa[j] * sq;
            Kg[r * P + lane + 32 * j] = ka[j] * sk;
        }
        if (lane == 0) bs[r] = r < L ? beta[(size_t)(t0 + r) * H + h] : 0.f;
    }
    __syncthreads();

    // 2. cumulative log-decay per channel and the decayed q/k (thread = channel).
    //    The Gram factors are referred to the midpoint B = b_last / 2 of the
    //    channel's decay range: Qg, Kg hold e^(b - B), Kd e^(B - b) (each within
    //    e^(|b_last| / 2)); the true Qg, Kg are these times mu = e^B, and
    //    Ke = Kd mu (b_last - B = B).
    if (tid < D) {
        const int d = tid;
        auto gate = [&](int r) {
            return scalar_gate ? g[(size_t)(t0 + r) * H + h] : g[((size_t)(t0 + r) * H + h) * D + d];
        };
        float tot = 0.f;
        for (int r = 0; r < L; ++r) tot += gate(r);
        const float B = 0.5f * tot;
        bool strong = false;
        float b = 0.f;
        for (int r = 0; r < kC; ++r) {
            if (r < L) b += gate(r);
            const float x = b - B;
            strong |= fabsf(x) > kMaxDecayExp;
            const float e = expf(fminf(x, kMaxDecayExp)), ei = expf(fminf(-x, kMaxDecayExp));
            const float kh = Kg[r * P + d];
            Qg[r * P + d] *= e;
            Kg[r * P + d] = kh * e;
            Kd[r * P + d] = kh * ei;
        }
        if (strong) record_status(st, (int32_t)KDA_ERR_UNSUPPORTED);
        const float m = expf(B);
        mu[d] = m;
        ho.gl[d] = m * m;
        for (int r = 0; r < kC; ++r) ho.Ke[r * D + d] = Kd[r * P + d] * m;
    }
    __syncthreads();

    for (int i = tid; i < kC * D; i += kThreads) ho.Qg[i] = Qg[(i / D) * P + (i % D)] * mu[i % D];

    // 3. Gram products: thread owns rows tr + 16a and columns ti + 16b (a, b < 4).
    {
        const int tr = tid >> 4, ti = tid & 15;
        float kk[4][4] = {}, qk[4][4] = {};
        for (int d = 0; d < D; ++d) {
            float kg[4], qg[4], kd[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                kg[a] = Kg[(tr + 16 * a) * P + d];
                qg[a] = Qg[(tr + 16 * a) * P + d];
                kd[a] = Kd[(ti + 16 * a) * P + d];
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    kk[a][c] += kg[a] * kd[c];
                    qk[a][c] += qg[a] * kd[c];
                }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int r = tr + 16 * a, i = ti + 16 * c;
                Lm[r * (kC + 1) + i] = (i < r) ? bs[r] * kk[a][c] : 0.f;
                ho.M[r * kC + i] = (i <= r) ? qk[a][c] : 0.f;
            }
    }
    __syncthreads();

    // 4. Tm = (I + Lm)^-1, one column per thread by forward substitution.
    if (tid < kC) {
        const int j = tid;
        for (int r = 0; r < kC; ++r) {
            float x = (r == j) ? 1.f : 0.f;
            if (r > j) {
                for (int i = j; i < r; ++i) x -= Lm[r * (kC + 1) + i] * Tm[i * (kC + 1) + j];
            }
            Tm[r * (kC + 1) + j] = x;
        }
    }
    __syncthreads();

    // 5. Wk = Tm diag(beta) Kg and Uv = Tm diag(beta) V (Tm is lower-triangular).
    for (int o = tid; o < kC * D; o += kThreads) {
        const int r = o / D, d = o % D;
        float wk = 0.f, uv = 0.f;
        for (int i = 0; i <= r; ++i) {
            const float t = Tm[r * (kC + 1) + i] * bs[i];
            wk += t * Kg[i * P + d];
            uv += t * Vs[i * P + d];
        }
        ho.Wk[o] = wk * mu[d];
        ho.Uv[o] = uv;
    }
}

// ---------------------------------------------------------------- K2
// One CTA per (sequence, head, 32-column block of Dv); serial over chunks.
constexpr int kBV = 32;

template <int D, typename T>
__global__ void __launch_bounds__(kThreads)
k2_simt_kernel(StateIO io, int N, int H, SeqTable tab, const float *__restrict__ handoff,
               T *__restrict__ out, const T *__restrict__ gate, Bounds bd)
{
    constexpr int P = D + 1;
    constexpr int NB = D / kBV;
    extern __shared__ float smem[];
    float *Ss = smem;                 // [D][kBV]   state block
    float *Ws = Ss + D * kBV;         // [C][kBV]   pseudo-values
    float *Wk = Ws + kC * kBV;        // [C][P]
    float *Qg = Wk + kC * P;          // [C][P]
    float *Ke = Qg + kC * P;          // [C][P]
    float *Ms = Ke + kC * P;          // [C][C+1]
    float *Us = Ms + kC * (kC + 1);   // [C][kBV]
    float *gl = Us + kC * kBV;        // [D]

    const int tid = threadIdx.x;
    const int jb = blockIdx.x % NB;
    const int h = (blockIdx.x / NB) % H;
    const int n = blockIdx.x / (NB * H);
    // this CTA's column block of the chain's initial and final states (dense
    // arrays or pool slots)
    const size_t DD = (size_t)D * D;
    int64_t is = io.init ? pool_slot(io.init_slots, n, io.pool) : -1;
    int64_t fs = io.fin ? pool_slot(io.final_slots, n, io.pool) : -1;
    if (is >= 0 && !dbg_in(is, bd.states, kDbgState)) is = -1;
    if (fs >= 0 && !dbg_in(fs, bd.states, kDbgState)) fs = -1;
    const float *init_blk = is >= 0 ? io.init + ((size_t)is * H + h) * DD + jb * kBV : nullptr;
    float *fin_blk = fs >= 0 ? io.fin + ((size_t)fs * H + h) * DD + jb * kBV : nullptr;
    const int stride = io.stride;

    for (int i = tid; i < D * kBV; i += kThreads) {
        const int d = i / kBV, j = i % kBV;
        Ss[i] = init_blk ? init_blk[(size_t)d * D + j] : 0.f;
    }
    const int c_begin = tab.chunk_off[n], c_end = tab.chunk_off[n + 1];
    const int seq_t0 = tab.cu[n], seq_t1 = tab.cu[n + 1];
    const int j = tid % kBV, rgrp = tid / kBV;   // rgrp in [0, 8)

    for (int gc = c_begin; gc < c_end; ++gc) {
        const int lc = gc - c_begin;
        const int t0 = seq_t0 + lc * kC;
        const int L = min(kC, seq_t1 - t0);
        if (!dbg_in((int64_t)gc * H + h, bd.records, kDbgRecord)) break;   // uniform over the CTA
        const int Lo = dbg_rows(t0, L, bd);   // output rows inside the token buffers (L but in a debug build)
        const float *p = handoff + ((size_t)gc * H + h) * handoff_floats(D);
        const float *hQg = p, *hWk = p + kC * D, *hUv = p + 2 * kC * D, *hKe = p + 3 * kC * D;
        const float *hM = p + 4 * kC * D, *hgl = hM + kC * kC;
        __syncthreads();
        for (int i = tid; i < kC * D; i += kThreads) {
            const int r = i / D, d = i % D;
            Wk[r * P + d] = hWk[i];
            Qg[r * P + d] = hQg[i];
            Ke[r * P + d] = hKe[i];
        }
        for (int i = tid; i < kC * kC; i += kThreads) Ms[(i / kC) * (kC + 1) + i % kC] = hM[i];
        for (int i = tid; i < kC * kBV; i += kThreads)
            Us[i] = hUv[(i / kBV) * D + jb * kBV + i % kBV];
        for (int i = tid; i < D; i += kThreads) gl[i] = hgl[i];
        __syncthreads();

        // W = Uv - Wk S0
        for (int r = rgrp; r < kC; r += kThreads / kBV) {
            float acc = Us[r * kBV + j];
            for (int d = 0; d < D; ++d) acc -= Wk[r * P + d] * Ss[d * kBV + j];
            Ws[r * kBV + j] = acc;
        }
        __syncthreads();
        // O = Qg S0 + M W
        for (int r = rgrp; r < Lo; r += kThreads / kBV) {
            float acc = 0.f;
            for (int d = 0; d < D; ++d) acc += Qg[r * P + d] * Ss[d * kBV + j];
            for (int i = 0; i <= r; ++i) acc += Ms[r * (kC + 1) + i] * Ws[i * kBV + j];
            const size_t oi = ((size_t)(t0 + r) * H + h) * D + jb * kBV + j;
            if (gate) acc /= 1.f + expf(-to_f32(gate[oi]));   // the fused output gate o sigmoid(z)
            out[oi] = from_f32<T>(acc);
        }
        __syncthreads();
        // S1 = Diag(gamma_last) S0 + Ke^T W
        for (int d = rgrp; d < D; d += kThreads / kBV) {
            float acc = gl[d] * Ss[d * kBV + j];
            for (int r = 0; r < L; ++r) acc += Ke[r * P + d] * Ws[r * kBV + j];
            Ss[d * kBV + j] = acc;
        }
        // checkpoint after every `stride` tokens of the sequence
        const int done = lc * kC + L;
        if (stride > 0 && io.ckpts && L == kC && done % stride == 0) {
            const int64_t jc = (int64_t)tab.ckpt_off[n] + done / stride - 1;
            const int64_t ps = jc < io.capacity ? pool_slot(io.ckpt_slots, jc, io.pool) : -1;
            if (ps >= 0 && dbg_in(ps, bd.ckpts, kDbgCkpt)) {
                __syncthreads();
                float *dst = io.ckpts + ((size_t)ps * H + h) * DD + jb * kBV;
                for (int i = tid; i < D * kBV; i += kThreads)
                    dst[(size_t)(i / kBV) * D + i % kBV] = Ss[i];
            }
        }
    }
    __syncthreads();
    if (fin_blk)
        for (int i = tid; i < D * kBV; i += kThreads) fin_blk[(size_t)(i / kBV) * D + i % kBV] = Ss[i];
}

template <int D, typename T>
cudaError_t launch_simt_t(const PrefillArgs &a)
{
    constexpr int P = D + 1;
    const size_t sm1 = sizeof(float) * ((size_t)4 * kC * P + 2 * kC * (kC + 1) + kC + D);
    const size_t sm2 = sizeof(float) * ((size_t)D * kBV + kC * kBV + 3 * kC * P +
                                        kC * (kC + 1) + kC * kBV + D);
    cudaError_t e;
    e = cudaFuncSetAttribute(k1_simt_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm1);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k2_simt_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm2);
    if (e != cudaSuccess) return e;
    if (a.max_chunks > 0) {
        dim3 g1((unsigned)a.max_chunks, (unsigned)a.H);
        k1_simt_kernel<D, T><<<g1, kThreads, sm1, a.stream>>>(
            (const T *)a.q, (const T *)a.k, (const T *)a.v, a.g, a.beta, a.N, a.H, a.tab,
            (float *)a.handoff, a.scalar_gate ? 1 : 0, a.status, a.conv_w, a.conv_width, a.conv_silu,
            (const T *)a.conv_in, a.bounds);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const unsigned g2 = (unsigned)((size_t)a.N * a.H * (D / kBV));
    k2_simt_kernel<D, T><<<g2, kThreads, sm2, a.stream>>>(state_io(a), a.N, a.H, a.tab,
                                                           (const float *)a.handoff, (T *)a.out, (const T *)a.gate,
                                                           a.bounds);
    return cudaGetLastError();
}

}  // namespace

size_t simt_handoff_bytes_per_chunk(int D, int /*C*/) { return sizeof(float) * handoff_floats(D); }

// The convolution state after each sequence: its last W - 1 raw q, k, v rows
// (oldest first), reaching into the history before it when the sequence is
// shorter.  One CTA per (sequence, head); each thread owns whole columns
// (tensor, channel) and reads them before writing, so the output may be the
// history buffer itself.
template <typename T>
__global__ void conv_tail_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                                 const T *conv_in, T *conv_out, int N, int H, int D, int W, SeqTable tab,
                                 Bounds bd)
{
    const int n = blockIdx.x / H, h = blockIdx.x % H;
    const int len = tab.cu[n + 1] - tab.cu[n];
    for (int col = threadIdx.x; col < 3 * D; col += blockDim.x) {
        const int t = col / D, c = col % D;
        const T *x = t == 0 ? q : t == 1 ? k : v;
        T vals[kConvTaps - 1];
        for (int j = 0; j < W - 1; ++j) {
            const int p = len - (W - 1) + j;   // position in the sequence
            if (p >= 0)
                vals[j] = dbg_in((int64_t)tab.cu[n] + p, bd.tokens, kDbgTokenRow)
                              ? x[((size_t)(tab.cu[n] + p) * H + h) * D + c] : from_f32<T>(0.f);
            else if (conv_in)
                vals[j] = conv_in[((((size_t)n * 3 + t) * (W - 1) + (W - 1 + p)) * H + h) * D + c];
            else vals[j] = from_f32<T>(0.f);
        }
        for (int j = 0; j < W - 1; ++j) conv_out[((((size_t)n * 3 + t) * (W - 1) + j) * H + h) * D + c] = vals[j];
    }
}

cudaError_t launch_conv_tail(const PrefillArgs &a)
{
    if (a.conv_width <= 1) return cudaSuccess;
    const unsigned grid = (unsigned)((size_t)a.N * a.H);
    if (a.dtype == KDA_DTYPE_BF16)
        conv_tail_kernel<__nv_bfloat16><<<grid, 128, 0, a.stream>>>(
            (const __nv_bfloat16 *)a.q, (const __nv_bfloat16 *)a.k, (const __nv_bfloat16 *)a.v,
            (const __nv_bfloat16 *)a.conv_in, (__nv_bfloat16 *)a.conv_out, a.N, a.H, a.D, a.conv_width, a.tab,
            a.bounds);
    else
        conv_tail_kernel<float><<<grid, 128, 0, a.stream>>>((const float *)a.q, (const float *)a.k,
                                                             (const float *)a.v, (const float *)a.conv_in,
                                                             (float *)a.conv_out, a.N, a.H, a.D, a.conv_width,
                                                             a.tab, a.bounds);
    return cudaGetLastError();
}

cudaError_t launch_seq_table(const PrefillArgs &a)
{
    seq_table_kernel<<<1, 32, 0, a.stream>>>(a.cu_seqlens, a.N, a.T, a.C, a.ckpt_stride,
                                             a.ckpt_capacity, a.seq_cap_chunks, a.tab, a.status);
    return cudaGetLastError();
}

cudaError_t launch_prefill_simt(const PrefillArgs &a)
{
    if (a.D == 128)
        return a.dtype == KDA_DTYPE_BF16 ? launch_simt_t<128, __nv_bfloat16>(a)
                                         : launch_simt_t<128, float>(a);
    return a.dtype == KDA_DTYPE_BF16 ? launch_simt_t<64, __nv_bfloat16>(a)
                                     : launch_simt_t<64, float>(a);
}

KDA_DBG_TAKE(dbg_take_prefill_simt)

}  // namespace kda
