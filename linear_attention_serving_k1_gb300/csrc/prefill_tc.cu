// prefill_tc.cu -- chunked KDA prefill on the sm_103a tensor cores (tcgen05,
// accumulators in TMEM), bf16 q/k/v, fp32 gates, fp32 state, D = 128, C = 64.
//
// Method: the token recurrence unrolled into chunks (page "Kimi K3
// reconstructs long-context inference efficiency through KDA, cross-depth
// attention, and latent expert routing", section "Methodology notes", item
// "System optimization: FlashKDA": K1 tensor preparation in parallel over
// chunks, K2 blockwise recurrence) with the UT transform of the zsxq post on
// SemiAnalysis' Kimi K3 analysis, section "一、Kimi Delta Attention（KDA）".
//
// Per chunk (rows r < 64, start state S, d = key channel, e = value column):
//   K1  qh, kh; b = inclusive cumsum of g; Qg = qh e^b, Kg = kh e^b,
//       Kd = kh e^-b, Ke = kh e^(b_last - b), gamma = e^b_last
//       G  = [Kg; Qg] Kd^T                        (one M=128 MMA)
//       L  = strict-lower(diag(beta) Kg Kd^T), Mc = incl-lower(Qg Kd^T)
//       T  = (I + L)^-1                            (fp32, blocked, CUDA cores)
//       Wk = T diag(beta) Kg, Uv = T diag(beta) V   (MMAs)
//       A' = -Ke^T Wk,  Q' = Qg - Mc Wk             (MMAs)
//   K2  S_next = Diag(gamma) S + A' S + Ke^T Uv     (fp32 state, one MMA
//                                                    on the serial path)
//       O      = Q' S + Mc Uv
// which is W = Uv - Wk S, O = Qg S + Mc W, S_next = Diag(gamma) S + Ke^T W
// with W eliminated: the serial chain carries one state-dependent MMA per
// chunk instead of two.
//
// Precision: fp32 state and accumulation throughout; tensor-core operands are
// tf32 for the Gram product of K1 and f16 for every other product (values
// of v and of the state must stay within the f16 range, |x| < 65504).
//
// K1 writes, per (chunk, head), one 90,624-byte record holding the K2 operand
// tiles already in the tensor-core shared-memory layout (no-swizzle K-major
// core matrices), so K2 moves each record into shared memory with a single
// bulk (TMA) copy.
#include "kda_common.cuh"
#include "tc.cuh"

#include <cuda_fp16.h>

namespace kda {
namespace {

using namespace tc;
typedef __nv_bfloat16 bf16;

constexpr int kC = 64;
constexpr int kD = 128;

// ------------------------------------------------------------ record layout
// A'  : B operand, rows d (128) x K = d' (128)   LBO 128, SBO 2048
// Q'  : B operand, rows r (64)  x K = d (128)    LBO 128, SBO 2048
// Uv^T: A operand, rows e (128) x K = r (64)     LBO 128, SBO 1024
// Ke^T: B operand, rows d (128) x K = r (64)     LBO 128, SBO 1024
// Mc  : B operand, rows r (64)  x K = i (64)     LBO 128, SBO 1024
// gamma: fp32 [128]
constexpr uint32_t REC_AP = 0;
constexpr uint32_t REC_QP = 32768;
constexpr uint32_t REC_UVT = 49152;
constexpr uint32_t REC_KET = 65536;
constexpr uint32_t REC_M = 81920;
constexpr uint32_t REC_G = 90112;
constexpr uint32_t REC_BYTES = 90624;
constexpr uint32_t SBO_K128 = 2048;   // 8-row group stride when K = 128 (K-inner packing)
constexpr uint32_t SBO_K64 = 1024;    // ... when K = 64
constexpr uint32_t LBO_KIN = 128;     // K-inner packing: core matrices along K are adjacent

// ------------------------------------------------------------ small helpers
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ int find_seq_tc(const int32_t *chunk_off, int N, int gc)
{
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (chunk_off[mid] <= gc) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ void record_timeout(DevStatus *st)
{
    atomicExch(&st->code, (int32_t)KDA_ERR_TIMEOUT);
}

// Polls `bar` for phase `parity`; gives up after a bounded number of polls, or
// early when another role of the CTA has flagged an abort.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag)
{
    for (uint32_t i = 0; i < (1u << 22); ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 1023u) == 1023u && *abort_flag) return false;
    }
    return false;
}

constexpr uint32_t kWaitLimit = 1u << 22;

// ============================================================ K1
// One CTA (128 threads) per (chunk, head).  The Gram product G = [Kg; Qg] Kd^T
// runs as tf32 (its decayed factors e^{+-b} need the fp32 exponent range);
// every other product takes f16 operands (11 significant bits: the bf16
// rounding of 8 bits was measured to put the max output error of long
// sequences past 2e-2 of the rms, f16/tf32 operands keep it near 3e-3).
//
// Shared memory map (bytes).  The first 73,728 bytes (Kd and the Kg half of
// [Kg; Qg]) are free once G is computed and are reused by the second phase.
constexpr uint32_t K1_KD = 0;            // tf32 Kd: rows i 64 x K = d 128, K-inner, LBO 144
constexpr uint32_t K1_GA = 36864;        // tf32 [Kg; Qg]: rows 128 x K = d 128, K-inner, LBO 144
constexpr uint32_t K1_F32_LBO = 144;     // 128 + 16: conflict-free scattered 4-byte stores
constexpr uint32_t K1_F32_SBO = 32 * K1_F32_LBO;
constexpr uint32_t K1_KGT = K1_GA + 16 * K1_F32_SBO;   // f16 Kg^T: rows d x K = i (128 x 64)
constexpr uint32_t K1_VT = K1_KGT + 16384;             // f16 V^T : rows e x K = i
constexpr uint32_t K1_KET = K1_VT + 16384;             // f16 Ke^T: rows d x K = r
constexpr uint32_t K1_SMEM = K1_KET + 16384;
// second phase, inside [0, 73728)
constexpr uint32_t K1_LM = 0;            // fp32 [64][65]  L (strict lower, beta-scaled)
constexpr uint32_t K1_TM = 16640;        // fp32 [64][65]  T = (I + L)^-1
constexpr uint32_t K1_XS = 33280;        // fp32 [3][16][17] scratch of the blocked inverse
constexpr uint32_t K1_TB = 36864;        // f16 T diag(beta): rows r x K = i (64 x 64)
constexpr uint32_t K1_MC = 45056;        // f16 Mc: rows r x K = i (64 x 64)
constexpr uint32_t K1_WKT = 53248;       // f16 Wk^T: rows d x K = r (128 x 64)
static_assert(K1_WKT + 16384 <= K1_GA + 8 * K1_F32_SBO, "second phase must stay in the freed region");

// TMEM columns (256 allocated)
constexpr uint32_t T1_G = 0, T1_W1 = 64, T1_W2 = 128, T1_AP = 0, T1_QP = 128;

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__global__ void __launch_bounds__(128, 1)
k1_tc_kernel(const bf16 *__restrict__ q, const bf16 *__restrict__ k, const bf16 *__restrict__ v,
             const float *__restrict__ g, const float *__restrict__ beta, int N, int H, SeqTable tab,
             uint8_t *__restrict__ handoff, DevStatus *st)
{
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ uint64_t mbar;
    __shared__ uint32_t tmem_sh;
    __shared__ float rq[kC], rk[kC], bs[kC];

    const int gc = blockIdx.x, h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (gc >= tab.chunk_off[N]) return;   // uniform across the CTA, before any allocation
    const int n = find_seq_tc(tab.chunk_off, N, gc);
    const int t0 = tab.cu[n] + (gc - tab.chunk_off[n]) * kC;
    const int L = min(kC, tab.cu[n + 1] - t0);
    uint8_t *rec = handoff + ((size_t)gc * H + h) * REC_BYTES;

    if (warp == 0) {
        tmem_alloc(&tmem_sh, 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&mbar, 1);
        fence_mbar_init();
    }

    // 1. row norms of q and k (warp w: rows 16w..16w+15), beta
    for (int rr = 0; rr < 16; ++rr) {
        const int r = warp * 16 + rr;
        float sq = 0.f, sk = 0.f;
        if (r < L) {
            const size_t base = ((size_t)(t0 + r) * H + h) * kD + lane * 4;
            const uint2 qa = *reinterpret_cast<const uint2 *>(q + base);
            const uint2 ka = *reinterpret_cast<const uint2 *>(k + base);
            float a0 = bf_lo(qa.x), a1 = bf_hi(qa.x), a2 = bf_lo(qa.y), a3 = bf_hi(qa.y);
            float c0 = bf_lo(ka.x), c1 = bf_hi(ka.x), c2 = bf_lo(ka.y), c3 = bf_hi(ka.y);
            sq = a0 * a0 + a1 * a1 + a2 * a2 + a3 * a3;
            sk = c0 * c0 + c1 * c1 + c2 * c2 + c3 * c3;
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        if (lane == 0) {
            rq[r] = r < L ? rsqrtf(sq + 1e-6f) : 0.f;
            rk[r] = r < L ? rsqrtf(sk + 1e-6f) : 0.f;
        }
    }
    if (tid < kC) bs[tid] = tid < L ? beta[(size_t)(t0 + tid) * H + h] : 0.f;
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = tmem_sh;

    // 2. thread d = tid: cumulative log-decay, then the decayed q/k operands
    const int d = tid;
    float b[kC];
    {
        float acc = 0.f;
#pragma unroll
        for (int r = 0; r < kC; ++r) {
            if (r < L) acc += g[((size_t)(t0 + r) * H + h) * kD + d];
            b[r] = acc;
        }
    }
    const float bl = b[kC - 1];
    const float gl = __expf(bl);
    reinterpret_cast<float *>(rec + REC_G)[d] = gl;
#pragma unroll
    for (int r8 = 0; r8 < kC; r8 += 8) {
        uint32_t pkg[4], pv[4], pke[4];
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            float kgv[2], vv2[2], kev[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int r = r8 + j + u;
                float qv = 0.f, kv = 0.f, vv = 0.f;
                if (r < L) {
                    const size_t base = ((size_t)(t0 + r) * H + h) * kD + d;
                    qv = __bfloat162float(q[base]);
                    kv = __bfloat162float(k[base]);
                    vv = __bfloat162float(v[base]);
                }
                const float qh = qv * rq[r], kh = kv * rk[r];
                const float e = __expf(b[r]), ei = __expf(-b[r]);
                const float Kg = kh * e, Qg = qh * e, Kd = kh * ei;
                *reinterpret_cast<float *>(sm + K1_GA + kmaj_off4(r, d, K1_F32_LBO, K1_F32_SBO)) = round_tf32(Kg);
                *reinterpret_cast<float *>(sm + K1_GA + kmaj_off4(64 + r, d, K1_F32_LBO, K1_F32_SBO)) = round_tf32(Qg);
                *reinterpret_cast<float *>(sm + K1_KD + kmaj_off4(r, d, K1_F32_LBO, K1_F32_SBO)) = round_tf32(Kd);
                kgv[u] = Kg;
                vv2[u] = vv;
                kev[u] = Kd * gl;   // kh * exp(b_last - b_r)
            }
            pkg[j / 2] = pack_f16x2(kgv[0], kgv[1]);
            pv[j / 2] = pack_f16x2(vv2[0], vv2[1]);
            pke[j / 2] = pack_f16x2(kev[0], kev[1]);
        }
        *reinterpret_cast<uint4 *>(sm + K1_KGT + kmaj_off(d, r8, LBO_KIN, SBO_K64)) = make_uint4(pkg[0], pkg[1], pkg[2], pkg[3]);
        *reinterpret_cast<uint4 *>(sm + K1_VT + kmaj_off(d, r8, LBO_KIN, SBO_K64)) = make_uint4(pv[0], pv[1], pv[2], pv[3]);
        *reinterpret_cast<uint4 *>(sm + K1_KET + kmaj_off(d, r8, LBO_KIN, SBO_K64)) = make_uint4(pke[0], pke[1], pke[2], pke[3]);
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // 3. G = [Kg; Qg] Kd^T  (tf32, M = 128, N = 64, K = 128: 16 instructions of K = 8)
    if (tid == 0) {
        const uint32_t idesc = idesc_tf32(128, 64);
        const uint32_t a0 = smem_u32(sm + K1_GA), b0 = smem_u32(sm + K1_KD);
#pragma unroll
        for (int ks = 0; ks < kD / 8; ++ks)
            mma_tf32(tm + T1_G, make_desc(a0 + ks * 2 * K1_F32_LBO, K1_F32_LBO, K1_F32_SBO),
                     make_desc(b0 + ks * 2 * K1_F32_LBO, K1_F32_LBO, K1_F32_SBO), idesc, ks > 0);
        mma_commit(&mbar);
    }
    bool ok = mbar_wait_bounded(&mbar, 0, kWaitLimit);
    fence_after_sync();
    __syncthreads();   // every thread has seen G complete: the first-phase region may be reused

    // 4. read G: warps 0-1 hold rows of Kg Kd^T (-> L), warps 2-3 rows of Qg Kd^T (-> Mc)
    float *Lm = reinterpret_cast<float *>(sm + K1_LM);
    float *Tm = reinterpret_cast<float *>(sm + K1_TM);
    float *Xs = reinterpret_cast<float *>(sm + K1_XS);
    if (ok) {
        float gv[64];
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
            float t16[16];
            tmem_ld16(tm + ((uint32_t)(32 * warp) << 16) + T1_G + c, t16);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) gv[c + i] = t16[i];
        }
        if (warp < 2) {
            const int r = tid;
            const float br = bs[r];
#pragma unroll
            for (int i = 0; i < 64; ++i) Lm[r * 65 + i] = (i < r) ? br * gv[i] : 0.f;
        } else {
            const int r = tid - 64;
#pragma unroll
            for (int i8 = 0; i8 < 64; i8 += 8) {
                uint32_t p[4];
#pragma unroll
                for (int j = 0; j < 8; j += 2)
                    p[j / 2] = pack_f16x2((i8 + j <= r) ? gv[i8 + j] : 0.f,
                                          (i8 + j + 1 <= r) ? gv[i8 + j + 1] : 0.f);
                const uint4 val = make_uint4(p[0], p[1], p[2], p[3]);
                *reinterpret_cast<uint4 *>(sm + K1_MC + kmaj_off(r, i8, LBO_KIN, SBO_K64)) = val;
                *reinterpret_cast<uint4 *>(rec + REC_M + kmaj_off(r, i8, LBO_KIN, SBO_K64)) = val;
            }
        }
    }
    __syncthreads();

    // 5. T = (I + L)^-1, blocked by 16: diagonal blocks by forward substitution,
    //    then T_ab = -T_aa * sum_{k=b}^{a-1} L_ak T_kb by block distance.
    if (tid < 64) {
        const int blk = tid >> 4, c = tid & 15, col = 16 * blk + c;
        for (int rr = 0; rr < 16; ++rr) {
            const int r = 16 * blk + rr;
            float x = (rr == c) ? 1.f : 0.f;
            for (int i = col; i < r; ++i) x -= Lm[r * 65 + i] * Tm[i * 65 + col];
            Tm[r * 65 + col] = (rr >= c) ? x : 0.f;
        }
    } else {
        for (int idx = tid - 64; idx < 64 * 64; idx += 64) {
            const int r = idx >> 6, j = idx & 63;
            if ((j >> 4) > (r >> 4)) Tm[r * 65 + j] = 0.f;
        }
    }
    __syncthreads();
    for (int lvl = 1; lvl < 4; ++lvl) {
        const int nb = 4 - lvl;
        for (int idx = tid; idx < nb * 256; idx += 128) {
            const int bb = idx >> 8, i = (idx >> 4) & 15, j = idx & 15, a = bb + lvl;
            float s = 0.f;
            for (int kk = bb; kk < a; ++kk)
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    s += Lm[(16 * a + i) * 65 + 16 * kk + m] * Tm[(16 * kk + m) * 65 + 16 * bb + j];
            Xs[(bb * 16 + i) * 17 + j] = s;
        }
        __syncthreads();
        for (int idx = tid; idx < nb * 256; idx += 128) {
            const int bb = idx >> 8, i = (idx >> 4) & 15, j = idx & 15, a = bb + lvl;
            float s = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) s += Tm[(16 * a + i) * 65 + 16 * a + m] * Xs[(bb * 16 + m) * 17 + j];
            Tm[(16 * a + i) * 65 + 16 * bb + j] = -s;
        }
        __syncthreads();
    }

    // 6. T diag(beta) -> f16 operand (rows r, K = i)
    {
        const int r = tid >> 1, i0 = (tid & 1) * 32;
#pragma unroll
        for (int i8 = 0; i8 < 32; i8 += 8) {
            uint32_t p[4];
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                const int i = i0 + i8 + j;
                p[j / 2] = pack_f16x2(i <= r ? Tm[r * 65 + i] * bs[i] : 0.f,
                                      i + 1 <= r ? Tm[r * 65 + i + 1] * bs[i + 1] : 0.f);
            }
            *reinterpret_cast<uint4 *>(sm + K1_TB + kmaj_off(r, i0 + i8, LBO_KIN, SBO_K64)) =
                make_uint4(p[0], p[1], p[2], p[3]);
        }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // 7. Wk^T = Kg^T (T diag beta)^T and Uv^T = V^T (T diag beta)^T  (M = 128, N = 64, K = 64)
    if (tid == 0 && ok) {
        const uint32_t idesc = idesc_f16(128, 64);
        const uint32_t akg = smem_u32(sm + K1_KGT), av = smem_u32(sm + K1_VT), bt = smem_u32(sm + K1_TB);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            const uint64_t bd = make_desc(bt + ks * 256, LBO_KIN, SBO_K64);
            mma_f16(tm + T1_W1, make_desc(akg + ks * 256, LBO_KIN, SBO_K64), bd, idesc, ks > 0);
            mma_f16(tm + T1_W2, make_desc(av + ks * 256, LBO_KIN, SBO_K64), bd, idesc, ks > 0);
        }
        mma_commit(&mbar);
    }
    ok = ok && mbar_wait_bounded(&mbar, 1, kWaitLimit);
    fence_after_sync();

    // 8. Wk^T -> smem operand (rows d, K = r); Uv^T -> record (rows e, K = r)
    if (ok) {
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
            float w[16], u[16];
            tmem_ld16(tm + ((uint32_t)(32 * warp) << 16) + T1_W1 + c, w);
            tmem_ld16(tm + ((uint32_t)(32 * warp) << 16) + T1_W2 + c, u);
            tmem_ld_wait();
#pragma unroll
            for (int h8 = 0; h8 < 16; h8 += 8) {
                *reinterpret_cast<uint4 *>(sm + K1_WKT + kmaj_off(tid, c + h8, LBO_KIN, SBO_K64)) =
                    make_uint4(pack_f16x2(w[h8], w[h8 + 1]), pack_f16x2(w[h8 + 2], w[h8 + 3]),
                               pack_f16x2(w[h8 + 4], w[h8 + 5]), pack_f16x2(w[h8 + 6], w[h8 + 7]));
                *reinterpret_cast<uint4 *>(rec + REC_UVT + kmaj_off(tid, c + h8, LBO_KIN, SBO_K64)) =
                    make_uint4(pack_f16x2(u[h8], u[h8 + 1]), pack_f16x2(u[h8 + 2], u[h8 + 3]),
                               pack_f16x2(u[h8 + 4], u[h8 + 5]), pack_f16x2(u[h8 + 6], u[h8 + 7]));
            }
        }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // 9. A'acc = Ke^T Wk (M = 128, N = 128, K = 64); Q'acc = Mc Wk (M = 64, N = 128, K = 64)
    if (tid == 0 && ok) {
        const uint32_t ake = smem_u32(sm + K1_KET), amc = smem_u32(sm + K1_MC), bw = smem_u32(sm + K1_WKT);
        const uint32_t id128 = idesc_f16(128, 128), id64 = idesc_f16(64, 128);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            const uint64_t bd = make_desc(bw + ks * 256, LBO_KIN, SBO_K64);
            mma_f16(tm + T1_AP, make_desc(ake + ks * 256, LBO_KIN, SBO_K64), bd, id128, ks > 0);
            mma_f16(tm + T1_QP, make_desc(amc + ks * 256, LBO_KIN, SBO_K64), bd, id64, ks > 0);
        }
        mma_commit(&mbar);
    }
    ok = ok && mbar_wait_bounded(&mbar, 0, kWaitLimit);
    fence_after_sync();

    if (ok) {
        // 10. A' = -(Ke^T Wk) -> record (rows d, K = d')
#pragma unroll
        for (int c = 0; c < 128; c += 16) {
            float a[16];
            tmem_ld16(tm + ((uint32_t)(32 * warp) << 16) + T1_AP + c, a);
            tmem_ld_wait();
#pragma unroll
            for (int h8 = 0; h8 < 16; h8 += 8)
                *reinterpret_cast<uint4 *>(rec + REC_AP + kmaj_off(tid, c + h8, LBO_KIN, SBO_K128)) =
                    make_uint4(pack_f16x2(-a[h8], -a[h8 + 1]), pack_f16x2(-a[h8 + 2], -a[h8 + 3]),
                               pack_f16x2(-a[h8 + 4], -a[h8 + 5]), pack_f16x2(-a[h8 + 6], -a[h8 + 7]));
        }
        // 11. Q' = Qg - Mc Wk: the M = 64 accumulator puts row r = 16 w + l in lane 32 w + l (l < 16)
        const int r = 16 * warp + lane;
#pragma unroll
        for (int c = 0; c < 128; c += 16) {
            float a[16];
            tmem_ld16(tm + ((uint32_t)(32 * warp) << 16) + T1_QP + c, a);
            tmem_ld_wait();
            if (lane < 16) {
                float qg[16];
#pragma unroll
                for (int j4 = 0; j4 < 16; j4 += 4) {
                    const float4 t = *reinterpret_cast<const float4 *>(
                        sm + K1_GA + kmaj_off4(64 + r, c + j4, K1_F32_LBO, K1_F32_SBO));
                    qg[j4] = t.x; qg[j4 + 1] = t.y; qg[j4 + 2] = t.z; qg[j4 + 3] = t.w;
                }
#pragma unroll
                for (int h8 = 0; h8 < 16; h8 += 8)
                    *reinterpret_cast<uint4 *>(rec + REC_QP + kmaj_off(r, c + h8, LBO_KIN, SBO_K128)) =
                        make_uint4(pack_f16x2(qg[h8] - a[h8], qg[h8 + 1] - a[h8 + 1]),
                                   pack_f16x2(qg[h8 + 2] - a[h8 + 2], qg[h8 + 3] - a[h8 + 3]),
                                   pack_f16x2(qg[h8 + 4] - a[h8 + 4], qg[h8 + 5] - a[h8 + 5]),
                                   pack_f16x2(qg[h8 + 6] - a[h8 + 6], qg[h8 + 7] - a[h8 + 7]));
            }
        }
        // 12. Ke^T -> record (same layout as in shared memory)
        const uint4 *src = reinterpret_cast<const uint4 *>(sm + K1_KET);
        uint4 *dst = reinterpret_cast<uint4 *>(rec + REC_KET);
        for (int i = tid; i < 16384 / 16; i += 128) dst[i] = src[i];
    } else if (tid == 0) {
        record_timeout(st);
    }

    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tm, 256);
}

// ============================================================ K2
// One CTA per (sequence, head).  Warps 0-3: state / epilogue (thread e owns
// value column e of S, i.e. row e of S^T, in fp32 registers); warp 4: bulk
// copies of the K1 records (two stages); warp 5: tensor-core issue.
constexpr uint32_t K2_STAGE0 = 0;
constexpr uint32_t K2_SOP = 2 * REC_BYTES;            // f16 S^T: rows e x K = d (128 x 128)
constexpr uint32_t K2_SMEM = K2_SOP + 32768;
// TMEM columns (512 allocated): S accumulators (2 x 128), O accumulators (2 x 64)
constexpr uint32_t T2_S0 = 0, T2_O0 = 256;

__device__ __forceinline__ void write_sop(uint8_t *sop, int e, const float (&S)[kD])
{
#pragma unroll
    for (int d8 = 0; d8 < kD; d8 += 8)
        *reinterpret_cast<uint4 *>(sop + kmaj_off(e, d8, LBO_KIN, SBO_K128)) =
            make_uint4(pack_f16x2(S[d8], S[d8 + 1]), pack_f16x2(S[d8 + 2], S[d8 + 3]),
                       pack_f16x2(S[d8 + 4], S[d8 + 5]), pack_f16x2(S[d8 + 6], S[d8 + 7]));
}

__global__ void __launch_bounds__(192, 1)
k2_tc_kernel(const float *__restrict__ init_state, int N, int H, SeqTable tab,
             const uint8_t *__restrict__ handoff, bf16 *__restrict__ out,
             float *__restrict__ final_state, float *__restrict__ ckpts, int stride,
             int64_t capacity, DevStatus *st)
{
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ uint64_t full[2], empty[2], sdone[2], ofree[2], sready;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = blockIdx.x / H, h = blockIdx.x % H;
    const int c_begin = tab.chunk_off[n], nch = tab.chunk_off[n + 1] - c_begin;
    const int seq_t0 = tab.cu[n], seq_t1 = tab.cu[n + 1];

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1 + 128);   // MMA commit + every state thread
            mbar_init(&sdone[s], 1);
            mbar_init(&ofree[s], 128);
        }
        mbar_init(&sready, 128);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_sh, 512);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = tmem_sh;
    volatile int *abort_v = &abort_flag;

    if (warp < 4) {
        // ---------------------------------------------------------- state role
        const int e = tid;
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        float S[kD];
        const size_t sbase = ((size_t)n * H + h) * kD * kD;
#pragma unroll
        for (int d = 0; d < kD; ++d) S[d] = init_state ? init_state[sbase + (size_t)d * kD + e] : 0.f;
        write_sop(sm + K2_SOP, e, S);
        fence_async_smem();
        mbar_arrive(&sready);
        bool alive = true;
        for (int c = 0; c < nch && alive; ++c) {
            const int s = c & 1;
            if (!wait_or_abort(&sdone[s], (c >> 1) & 1, abort_v)) {
                alive = false;
                break;
            }
            fence_after_sync();
            const float *gam = reinterpret_cast<const float *>(sm + K2_STAGE0 + s * REC_BYTES + REC_G);
#pragma unroll
            for (int c32 = 0; c32 < kD; c32 += 32) {
                float a0[16], a1[16];
                tmem_ld16(tm + lane_base + T2_S0 + s * 128 + c32, a0);
                tmem_ld16(tm + lane_base + T2_S0 + s * 128 + c32 + 16, a1);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    S[c32 + j] = gam[c32 + j] * S[c32 + j] + a0[j];
                    S[c32 + 16 + j] = gam[c32 + 16 + j] * S[c32 + 16 + j] + a1[j];
                }
            }
            write_sop(sm + K2_SOP, e, S);
            fence_async_smem();
            fence_before_sync();
            mbar_arrive(&sready);
            mbar_arrive(&empty[s]);            // this thread is done with the stage's gamma

            // output rows of this chunk
            const int t0 = seq_t0 + c * kC;
            const int L = min(kC, seq_t1 - t0);
#pragma unroll
            for (int c16 = 0; c16 < kC; c16 += 16) {
                float o[16];
                tmem_ld16(tm + lane_base + T2_O0 + s * 64 + c16, o);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (c16 + j < L) out[((size_t)(t0 + c16 + j) * H + h) * kD + e] = __float2bfloat16_rn(o[j]);
            }
            fence_before_sync();
            mbar_arrive(&ofree[s]);

            // checkpoint after every `stride` tokens of the sequence
            const int done = c * kC + L;
            if (stride > 0 && ckpts && L == kC && done % stride == 0) {
                const int64_t slot = (int64_t)tab.ckpt_off[n] + done / stride - 1;
                if (slot < capacity) {
                    float *dst = ckpts + ((size_t)slot * H + h) * kD * kD + e;
#pragma unroll
                    for (int d = 0; d < kD; ++d) dst[(size_t)d * kD] = S[d];
                }
            }
        }
        if (!alive) {
            *abort_v = 1;
            if (tid == 0) record_timeout(st);
        } else if (final_state) {
#pragma unroll
            for (int d = 0; d < kD; ++d) final_state[sbase + (size_t)d * kD + e] = S[d];
        }
    } else if (warp == 4) {
        // ---------------------------------------------------------- bulk-copy role
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nch; ++c) {
                const int s = c & 1;
                if (c >= 2 && !wait_or_abort(&empty[s], ((c - 2) >> 1) & 1, abort_v)) {
                    *abort_v = 1;
                    record_timeout(st);
                    break;
                }
                mbar_arrive_expect_tx(&full[s], REC_BYTES);
                bulk_g2s(sm + K2_STAGE0 + s * REC_BYTES,
                         handoff + ((size_t)(c_begin + c) * H + h) * REC_BYTES, REC_BYTES, &full[s]);
                issued = c + 1;
            }
            // Never leave a copy in flight: wait for the last (up to two) copies.
            for (int c = max(0, issued - 2); c < issued; ++c)
                mbar_wait_bounded(&full[c & 1], (c >> 1) & 1, kWaitLimit);
        }
    } else {
        // ---------------------------------------------------------- MMA role
        if (lane == 0) {
            const uint32_t sop = smem_u32(sm + K2_SOP);
            const uint32_t id_s = idesc_f16(128, 128), id_o = idesc_f16(128, 64);
            for (int c = 0; c < nch; ++c) {
                const int s = c & 1;
                if (!wait_or_abort(&full[s], (c >> 1) & 1, abort_v) ||
                    (c >= 2 && !wait_or_abort(&ofree[s], ((c - 2) >> 1) & 1, abort_v))) {
                    *abort_v = 1;
                    record_timeout(st);
                    break;
                }
                fence_after_sync();
                const uint32_t stg = smem_u32(sm + K2_STAGE0 + s * REC_BYTES);
                const uint32_t dS = tm + T2_S0 + s * 128, dO = tm + T2_O0 + s * 64;
                // state-independent part: Ke^T Uv -> S acc, Mc Uv -> O acc
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t a = make_desc(stg + REC_UVT + ks * 256, LBO_KIN, SBO_K64);
                    mma_f16(dS, a, make_desc(stg + REC_KET + ks * 256, LBO_KIN, SBO_K64), id_s, ks > 0);
                    mma_f16(dO, a, make_desc(stg + REC_M + ks * 256, LBO_KIN, SBO_K64), id_o, ks > 0);
                }
                if (!wait_or_abort(&sready, c & 1, abort_v)) {
                    *abort_v = 1;
                    record_timeout(st);
                    break;
                }
                fence_after_sync();
                // state-dependent part: S acc += S^T A'^T, O acc += S^T Q'^T
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t a = make_desc(sop + ks * 256, LBO_KIN, SBO_K128);
                    mma_f16(dS, a, make_desc(stg + REC_AP + ks * 256, LBO_KIN, SBO_K128), id_s, 1);
                    mma_f16(dO, a, make_desc(stg + REC_QP + ks * 256, LBO_KIN, SBO_K128), id_o, 1);
                }
                mma_commit(&sdone[s]);
                mma_commit(&empty[s]);
            }
        }
    }

    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tm, 512);
}

}  // namespace

size_t tc_handoff_bytes_per_chunk() { return REC_BYTES; }

cudaError_t launch_prefill_tc(const PrefillArgs &a)
{
    cudaError_t e;
    e = cudaFuncSetAttribute(k1_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)K1_SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k2_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)K2_SMEM);
    if (e != cudaSuccess) return e;
    if (a.max_chunks > 0) {
        dim3 g1((unsigned)a.max_chunks, (unsigned)a.H);
        k1_tc_kernel<<<g1, 128, K1_SMEM, a.stream>>>(
            (const bf16 *)a.q, (const bf16 *)a.k, (const bf16 *)a.v, a.g, a.beta, a.N, a.H, a.tab,
            (uint8_t *)a.handoff, a.status);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    k2_tc_kernel<<<(unsigned)((size_t)a.N * a.H), 192, K2_SMEM, a.stream>>>(
        a.init_state, a.N, a.H, a.tab, (const uint8_t *)a.handoff, (bf16 *)a.out, a.final_state,
        a.ckpts, a.ckpt_stride, a.ckpt_capacity, a.status);
    return cudaGetLastError();
}

}  // namespace kda
