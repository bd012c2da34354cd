// decode.cu -- single-token KDA decode step, fp32 state updated in place.
//
// Page "Kimi K3 reconstructs long-context inference efficiency through KDA,
// cross-depth attention, and latent expert routing", section "Key data": a
// decode step costs about 7*D^2 FLOPs and 8*D^2 bytes per head, the bytes
// being one read and one write of the fp32 recurrent state.  The kernel is
// therefore a streaming pass over the state at HBM speed:
//
//   one CTA per (sequence, head); each warp streams whole 512-byte rows of S
//   as float4 (fully coalesced 128-bit loads); every element of S is read
//   once into registers, decayed there, used for both reductions, updated
//   from the same registers and written once.
//
//   S' = Diag(alpha) S                     (row scale, in registers)
//   sk = S'^T kh, sq = S'^T qh             (one pass, CTA reduction in smem)
//   u  = v - sk
//   o  = sq + beta (kh . qh) u             (= S_new^T qh, no second pass)
//   S_new = S' + beta kh u^T               (from registers, one write)
#include "kda_common.cuh"

namespace kda {
namespace {

// FUSED (single token, dense states): q, k, v pass through the short
// convolution with the sequence's history (conv_state, then advanced by the
// new raw rows) before the step, and the output through o * sigmoid(gate).
struct FusedIO {
    const float *conv_w;   // [3, W, H, D] or NULL
    int W, silu;
    void *conv_state;      // [N, 3, W - 1, H, D] of T, or NULL (zero history, nothing kept)
    const void *gate;      // [N, H, D] of T, or NULL
};

template <int D, typename T, int THREADS, bool MULTI, bool FUSED>
__device__ __forceinline__ void
decode_body(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
            const float *__restrict__ g, const float *__restrict__ beta,
            float *__restrict__ state, T *__restrict__ out, const int32_t *__restrict__ slots,
            int H, int64_t pool, int m_arg, const int32_t *__restrict__ commit, int32_t *status,
            int ahead, const Bounds &bd, const FusedIO &fz)
{
    const int m = MULTI ? m_arg : 1;   // a compile-time single token for plain decode
    constexpr int C4 = D / 4;            // float4 groups per state row
    constexpr int RPI = THREADS / C4;    // rows covered per pass of the CTA
    constexpr int RPT = D / RPI;         // rows per thread
    static_assert(THREADS % C4 == 0 && D % RPI == 0, "shape");
    constexpr int NW = THREADS / 32;

    const size_t head = blockIdx.x;      // (sequence n, head h) = n H + h
    const size_t n = head / (size_t)H, hh = head % (size_t)H;
    const int tid = threadIdx.x;
    const int c4 = tid % C4;
    const int r0 = tid / C4;

    // The state of (sequence n, head h) is block `head` of `state`, or, with a
    // slot table, block (slots[n], h) of a pool of `pool` slots; a slot outside
    // [0, pool) marks a padding row: no state access, zero output rows.
    size_t sblock = head;
    if (slots) {
        const int64_t sl = slots[n];
        if (sl < 0 || sl >= pool) {
            for (int t = 0; t < m; ++t)
                if (tid < D && dbg_in((int64_t)(n * m + t), bd.tokens, kDbgTokenRow))
                    out[((n * m + t) * H + hh) * D + tid] = from_f32<T>(0.f);
            return;
        }
        sblock = (size_t)sl * H + hh;
    }
    if (!dbg_in((int64_t)sblock, bd.states * H, kDbgState)) return;
    // The sequence's m tokens run one after another with the state in
    // registers; the state after `ncommit` of them is written back.
    const int ncommit = (MULTI && commit) ? min(max(commit[n], 0), m) : m;
    float4 *S = reinterpret_cast<float4 *>(state + sblock * (size_t)D * D);

    // Issue every state load first: RPT independent 16-byte loads per thread.
    float4 s[RPT];
#pragma unroll
    for (int j = 0; j < RPT; ++j) s[j] = __ldcs(S + (size_t)(r0 + j * RPI) * C4 + c4);

    // ... and bring the state of the CTA `ahead` positions later (a wave of one
    // CTA per SM) into L2 by line prefetches, so that the state stream keeps
    // going while CTAs reduce and write (calls about 7% shorter)
    if (ahead > 0 && blockIdx.x + (unsigned)ahead < gridDim.x) {
        const size_t head2 = blockIdx.x + (size_t)ahead;
        int64_t sb2 = (int64_t)head2;
        if (slots) {
            const int64_t sl2 = slots[head2 / (size_t)H];
            sb2 = (sl2 >= 0 && sl2 < pool) ? sl2 * H + (int64_t)(head2 % (size_t)H) : -1;
        }
        if (sb2 >= 0 && dbg_in(sb2, bd.states * H, kDbgState)) {
            const char *nx = reinterpret_cast<const char *>(state + (size_t)sb2 * D * D);
            for (int i = tid; i < D * D * 4 / 128; i += THREADS)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(nx + (size_t)i * 128));
        }
    }

    // Slots must be distinct: the head-0 CTA of sequence n compares its slot
    // with those of sequences 0 .. n-1 (while its state loads are in flight)
    // and reports a repeat in the caller's status word.
    if (slots && status && hh == 0) {
        const int32_t mine = slots[n];
        bool dup = false;
        for (size_t i = tid; i < n; i += THREADS) dup |= slots[i] == mine;
        if (dup) atomicCAS(status, 0, (int32_t)KDA_ERR_INVALID_ARG);
    }

    __shared__ float sh_qh[D], sh_kh[D], sh_a[D], sh_u[D];
    __shared__ float sh_part[3][NW];
    __shared__ float4 red_k[RPI][C4];
    __shared__ float4 red_q[RPI][C4];

    for (int t = 0; t < m; ++t) {
        // (debug build) a token row outside the token buffers: the whole CTA
        // skips the token (a uniform condition)
        if (!dbg_in((int64_t)(n * m + t), bd.tokens, kDbgTokenRow)) continue;
        const size_t tok = (n * m + t) * H + hh;   // token-head row of q, k, v, g, beta, out
        // Token vectors and the two L2 norms (fp32).
        float qv = 0.f, kv = 0.f, vconv = 0.f;
        if (tid < D) {
            qv = to_f32(q[tok * D + tid]);
            kv = to_f32(k[tok * D + tid]);
            sh_a[tid] = expf(g[tok * D + tid]);
            if constexpr (FUSED) {
                if (fz.conv_w) {
                    // x' = sum_{i < W-1} w[i] history[i] + w[W-1] x, then the history
                    // advances by the raw row (each thread owns its column of it)
                    T *cs = reinterpret_cast<T *>(fz.conv_state);
                    const float vraw = to_f32(v[tok * D + tid]);
                    float xs[3] = {qv, kv, vraw};
#pragma unroll
                    for (int t = 0; t < 3; ++t) {
                        float acc = fz.conv_w[(((size_t)t * fz.W + fz.W - 1) * H + hh) * D + tid] * xs[t];
                        float hist[3];
                        for (int i = 0; i < fz.W - 1; ++i) {
                            hist[i] = cs ? to_f32(cs[((((size_t)n * 3 + t) * (fz.W - 1) + i) * H + hh) * D + tid]) : 0.f;
                            acc += fz.conv_w[(((size_t)t * fz.W + i) * H + hh) * D + tid] * hist[i];
                        }
                        if (cs) {
                            for (int i = 0; i + 1 < fz.W - 1; ++i)
                                cs[((((size_t)n * 3 + t) * (fz.W - 1) + i) * H + hh) * D + tid] = from_f32<T>(hist[i + 1]);
                            if (fz.W > 1)
                                cs[((((size_t)n * 3 + t) * (fz.W - 1) + fz.W - 2) * H + hh) * D + tid] =
                                    t == 0 ? q[tok * D + tid] : t == 1 ? k[tok * D + tid] : v[tok * D + tid];
                        }
                        if (fz.silu) acc = acc / (1.f + expf(-acc));
                        xs[t] = acc;
                    }
                    qv = xs[0];
                    kv = xs[1];
                    vconv = xs[2];
                } else {
                    vconv = to_f32(v[tok * D + tid]);
                }
            }
        }
        float pq = warp_sum(qv * qv), pk = warp_sum(kv * kv), pqk = warp_sum(qv * kv);
        if ((tid & 31) == 0) {
            sh_part[0][tid >> 5] = pq;
            sh_part[1][tid >> 5] = pk;
            sh_part[2][tid >> 5] = pqk;
        }
        __syncthreads();
        float nq = 0.f, nk = 0.f, nqk = 0.f;
#pragma unroll
        for (int w = 0; w < (D + 31) / 32; ++w) {
            nq += sh_part[0][w];
            nk += sh_part[1][w];
            nqk += sh_part[2][w];
        }
        const float rq = rsqrtf(nq + 1e-6f), rk = rsqrtf(nk + 1e-6f);
        const float b = beta[tok];
        if (tid < D) {
            sh_qh[tid] = qv * rq;
            sh_kh[tid] = kv * rk;
        }
        __syncthreads();

        // Decay in registers and accumulate S'^T kh and S'^T qh.
        float4 ak = make_float4(0.f, 0.f, 0.f, 0.f), aq = ak;
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const int i = r0 + j * RPI;
            const float a = sh_a[i], kh = sh_kh[i], qh = sh_qh[i];
            s[j].x *= a; s[j].y *= a; s[j].z *= a; s[j].w *= a;
            ak.x += kh * s[j].x; ak.y += kh * s[j].y; ak.z += kh * s[j].z; ak.w += kh * s[j].w;
            aq.x += qh * s[j].x; aq.y += qh * s[j].y; aq.z += qh * s[j].z; aq.w += qh * s[j].w;
        }
        red_k[r0][c4] = ak;
        red_q[r0][c4] = aq;
        __syncthreads();

        if (tid < D) {
            const float *rk_ = reinterpret_cast<const float *>(&red_k[0][0]);
            const float *rq_ = reinterpret_cast<const float *>(&red_q[0][0]);
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int r = 0; r < RPI; ++r) {
                sk += rk_[r * D + tid];
                sq += rq_[r * D + tid];
            }
            const float u = (FUSED ? vconv : to_f32(v[tok * D + tid])) - sk;
            sh_u[tid] = u;
            const float kq = nqk * rq * rk;   // kh . qh
            float o = sq + b * kq * u;
            if constexpr (FUSED)
                if (fz.gate) o /= 1.f + expf(-to_f32(reinterpret_cast<const T *>(fz.gate)[tok * D + tid]));
            out[tok * D + tid] = from_f32<T>(o);
        }
        __syncthreads();

        const float4 u4 = reinterpret_cast<const float4 *>(sh_u)[c4];
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const int i = r0 + j * RPI;
            const float bk = b * sh_kh[i];
            s[j].x += bk * u4.x;
            s[j].y += bk * u4.y;
            s[j].z += bk * u4.z;
            s[j].w += bk * u4.w;
        }
        if (t + 1 == ncommit) {
#pragma unroll
            for (int j = 0; j < RPT; ++j) __stcs(S + (size_t)(r0 + j * RPI) * C4 + c4, s[j]);
        }
        __syncthreads();   // shared vectors are rewritten by the next token
    }
}

#define KDA_DECODE_PARAMS                                                                          \
    const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,                      \
        const float *__restrict__ g, const float *__restrict__ beta, float *__restrict__ state,      \
        T *__restrict__ out, const int32_t *__restrict__ slots, int H, int64_t pool, int m_arg,      \
        const int32_t *__restrict__ commit, int32_t *status, int ahead, Bounds bd
template <int D, typename T, int THREADS, bool MULTI, bool FUSED = false>
__global__ void __launch_bounds__(THREADS) decode_kernel(KDA_DECODE_PARAMS, FusedIO fz = FusedIO{})
{
    decode_body<D, T, THREADS, MULTI, FUSED>(q, k, v, g, beta, state, out, slots, H, pool, m_arg, commit, status,
                                             ahead, bd, fz);
}
// The single-token step (plain and paged decode) at 80 registers, so that
// three CTAs (192 KB of state loads in flight) share an SM instead of two: the
// few words it spills cost less than the third CTA gains (workload 3: 170.7
// against 172.7 us per step).
template <int D, typename T, int THREADS>
__global__ void __launch_bounds__(THREADS, 3) decode_kernel_3cta(KDA_DECODE_PARAMS)
{
    decode_body<D, T, THREADS, false, false>(q, k, v, g, beta, state, out, slots, H, pool, m_arg, commit, status,
                                             ahead, bd, FusedIO{});
}
#undef KDA_DECODE_PARAMS

template <int D, typename T>
cudaError_t launch_t(const void *q, const void *k, const void *v, const float *g,
                     const float *beta, float *state, void *out, int N, int H,
                     const int32_t *slots, int64_t pool, int m, const int32_t *commit, int32_t *status,
                     const Bounds &bd, cudaStream_t st)
{
    constexpr int THREADS = (D == 128) ? 256 : 128;
    const unsigned blocks = (unsigned)((size_t)N * H);
    const int ahead = (int)device_sm_count();
    if (m == 1 && !commit && D == 128)
        decode_kernel_3cta<D, T, THREADS><<<blocks, THREADS, 0, st>>>(
            (const T *)q, (const T *)k, (const T *)v, g, beta, state, (T *)out, slots, H, pool, 1, nullptr,
            status, ahead, bd);
    else if (m == 1 && !commit)
        decode_kernel<D, T, THREADS, false><<<blocks, THREADS, 0, st>>>(
            (const T *)q, (const T *)k, (const T *)v, g, beta, state, (T *)out, slots, H, pool, 1, nullptr,
            status, ahead, bd);
    else
        decode_kernel<D, T, THREADS, true><<<blocks, THREADS, 0, st>>>(
            (const T *)q, (const T *)k, (const T *)v, g, beta, state, (T *)out, slots, H, pool, m, commit,
            status, ahead, bd);
    return cudaGetLastError();
}

}  // namespace

template <int D, typename T>
cudaError_t launch_fused_t(const void *q, const void *k, const void *v, const float *g, const float *beta,
                           float *state, void *out, int N, int H, const DecodeFused &f, const Bounds &bd,
                           cudaStream_t st)
{
    constexpr int THREADS = (D == 128) ? 256 : 128;
    const FusedIO fz{f.conv_w, f.conv_width, f.conv_silu, f.conv_state, f.gate};
    decode_kernel<D, T, THREADS, false, true><<<(unsigned)((size_t)N * H), THREADS, 0, st>>>(
        (const T *)q, (const T *)k, (const T *)v, g, beta, state, (T *)out, nullptr, H, 0, 1, nullptr, nullptr,
        (int)device_sm_count(), bd, fz);
    return cudaGetLastError();
}

cudaError_t launch_decode_fused(const void *q, const void *k, const void *v, const float *g,
                                const float *beta, float *state, void *out, int N, int H, int D,
                                kda_dtype dtype, const DecodeFused &f, const Bounds &bd, cudaStream_t stream)
{
    if ((size_t)N * H == 0) return cudaSuccess;
    if (D == 128)
        return dtype == KDA_DTYPE_BF16
                   ? launch_fused_t<128, __nv_bfloat16>(q, k, v, g, beta, state, out, N, H, f, bd, stream)
                   : launch_fused_t<128, float>(q, k, v, g, beta, state, out, N, H, f, bd, stream);
    return dtype == KDA_DTYPE_BF16
               ? launch_fused_t<64, __nv_bfloat16>(q, k, v, g, beta, state, out, N, H, f, bd, stream)
               : launch_fused_t<64, float>(q, k, v, g, beta, state, out, N, H, f, bd, stream);
}

cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, float *state, void *out, int N, int H, int D,
                          kda_dtype dtype, const int32_t *slots, int64_t pool, int m,
                          const int32_t *commit, int32_t *status, const Bounds &bd, cudaStream_t stream)
{
    if ((size_t)N * H == 0 || m == 0) return cudaSuccess;
    if (D == 128)
        return dtype == KDA_DTYPE_BF16
                   ? launch_t<128, __nv_bfloat16>(q, k, v, g, beta, state, out, N, H, slots, pool, m, commit,
                                                  status, bd, stream)
                   : launch_t<128, float>(q, k, v, g, beta, state, out, N, H, slots, pool, m, commit, status,
                                          bd, stream);
    return dtype == KDA_DTYPE_BF16
               ? launch_t<64, __nv_bfloat16>(q, k, v, g, beta, state, out, N, H, slots, pool, m, commit, status,
                                             bd, stream)
               : launch_t<64, float>(q, k, v, g, beta, state, out, N, H, slots, pool, m, commit, status, bd, stream);
}

KDA_DBG_TAKE(dbg_take_decode)

}  // namespace kda
