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
//       T  = (I + L)^-1      (fp32, blocked: diagonal blocks on CUDA cores,
//                             merges on warp-level tensor-core MMAs)
//       Wk = T diag(beta) Kg, Uv = T diag(beta) V   (MMAs)
//       A' = -Ke^T Wk,  Q' = Qg - Mc Wk             (MMAs)
//   K2  [S_next - Diag(gamma) S | O] = [A' | Ke^T] [S; Uv] , [Q' | Mc] [S; Uv]
//       as one product per chunk (fp32 state and accumulation)
// which is W = Uv - Wk S, O = Qg S + Mc W, S_next = Diag(gamma) S + Ke^T W
// with W eliminated: the serial chain carries one state-dependent MMA group
// per chunk instead of two dependent ones, and the state-independent terms
// Ke^T Uv and Mc Uv ride in the same accumulator (their K-steps are issued
// before the state is ready).
//
// Precision: fp32 state and accumulation throughout; tensor-core operands are
// tf32 for the Gram product of K1 and f16 for every other product (values
// of k, v and of the state must stay within the f16 range, |x| < 65504).
//
// K1 writes, per (chunk, head), one record holding K2's operand tiles in the
// tensor-core shared-memory layout (no-swizzle K-major core matrices), moved
// into K2's shared memory by one bulk TMA copy, and gamma.
#include <atomic>
#include <type_traits>
#include "kda_common.cuh"
#include <algorithm>

#include "tc.cuh"

#include <cuda_fp16.h>
#include <stdio.h>

namespace kda {
namespace {

using namespace tc;
typedef __nv_bfloat16 bf16;

constexpr int kC = 64;
constexpr int kD = 128;

// ------------------------------------------------------------ record layout
// K2's B operand over K = d' (128): rows 0-127 A'[d][d'], rows 128-191 Q'[r][d];
// its B operand over K = r (64):    rows 0-127 Ke^T[d][r], rows 128-191 Mc[r][r'];
// its A operand over K = r:         rows e Uv^T[e][r];  then gamma, fp32 [128].
// f16, K-major, LBO 128; SBO 2048 for K = 128 and 1024 for K = 64.  With the
// L2 norms folded into scalars (see K1), the Ke^T rows hold k e^(b_last - b)
// un-normalised, Mc the rows of Qg Kd^T scaled by the query norm only, and
// Uv^T the columns of Uv scaled by the key norms: the products are the same.
constexpr uint32_t REC_AP = 0;          // A' (rows d), then Q' (rows r) at REC_QP
constexpr uint32_t REC_QP = 32768;
constexpr uint32_t REC_KM = 49152;      // Ke^T (rows d), then Mc (rows r) at REC_MC
constexpr uint32_t REC_MC = REC_KM + 16384;
constexpr uint32_t REC_UV = REC_KM + 24576;
constexpr uint32_t REC_G = REC_UV + 16384;
constexpr uint32_t REC_BYTES = REC_G + 512;
static_assert(REC_BYTES % 256 == 0, "record alignment");
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

constexpr float kLog2e = 1.4426950408889634f;   // log2(e)

// 2^x by the hardware's approximate base-2 exponential, results below the
// normal range flushed to zero (PTX ex2.approx.ftz.f32).
__device__ __forceinline__ float ex2_ftz(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void record_timeout(DevStatus *st)
{
    record_status(st, (int32_t)KDA_ERR_TIMEOUT);
}

// D += A B on the warp-level tensor-core path (m16n8k8, tf32 operands, fp32
// accumulation) with each operand split into its leading tf32 part and the
// fp32 remainder: the three products that matter (remainder terms first) give
// the sum to about 1e-6 relative instead of tf32's 1e-3.  Fragments of lane
// (g = lane / 4, t = lane % 4): a = A[g][t], A[g + 8][t], A[g][t + 4],
// A[g + 8][t + 4]; b = B[t][g], B[t + 4][g]; d = D[g][2t], D[g][2t + 1],
// D[g + 8][2t], D[g + 8][2t + 1].
__device__ __forceinline__ void mma_m16n8k8_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2])
{
    asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ void mma_tf32x3(float (&d)[4], const float (&a)[4], const float (&b)[2])
{
    uint32_t ah[4], al[4], bh[2], bl[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        ah[i] = __float_as_uint(a[i]) & 0xFFFFE000u;   // the bits a tf32 operand keeps
        al[i] = __float_as_uint(a[i] - __uint_as_float(ah[i]));
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        bh[i] = __float_as_uint(b[i]) & 0xFFFFE000u;
        bl[i] = __float_as_uint(b[i] - __uint_as_float(bh[i]));
    }
    mma_m16n8k8_tf32(d, al, bh);
    mma_m16n8k8_tf32(d, ah, bl);
    mma_m16n8k8_tf32(d, ah, bh);
}

// Polls `bar` for phase `parity`; gives up after `limit` polls, or early when
// another role of the CTA has flagged an abort.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              uint32_t limit)
{
    for (uint32_t i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 1023u) == 1023u && *abort_flag) return false;
    }
    return false;
}

// Polls allowed to the waits that drain a CTA's own tensor-core work and
// copies before it frees its TMEM and exits (independent of the call's wait
// limit: that work always completes, and must have before the exit).
constexpr uint32_t kDrainLimit = 1u << 22;

// ============================================================ K1
// One CTA (256 threads, two CTAs per SM) per (chunk, head).  The Gram product
// G = [Kg; Qg] Kd^T runs as tf32 (its decayed factors e^{+-b} need the fp32
// exponent range); every other product takes f16 operands (11 significant
// bits: the bf16 rounding of 8 bits was measured to put the max output error
// of long sequences past 2e-2 of the rms, f16/tf32 operands keep it near 3e-3).
//
// The L2 normalisation is folded into scalars instead of being applied to the
// operands first: with primes for un-normalised rows (Kg' = k e^b, ...) and
// rq, rk the inverse row norms of q and k,
//   L   = diag(beta rk) G'_kk diag(rk),     Mc = diag(rq) G'_qk diag(rk)
//   Wk  = T diag(beta rk) Kg',              Uv = T diag(beta) V
//   Ke^T Wk = Ke'^T diag(rk) Wk,  Mc Wk = Mc' diag(rk) Wk  (Mc' = diag(rq) G'_qk)
//   Ke^T Uv = Ke'^T diag(rk) Uv,  Mc Uv = Mc' diag(rk) Uv,   Qg = diag(rq) Qg'
// so the operands are built in one pass over the inputs, in two halves of the
// key channels (the Gram product accumulates over both), and the squared row
// norms are summed from the same registers.  Un-normalised f16 operands require |k| < 65504.
//
// Shared memory map (bytes).  [0, 55296) holds one key-channel half of the
// tf32 Gram operands and is reused by the later phases.
constexpr uint32_t K1_F32_LBO = 144;                   // 128 + 16: conflict-free 8-byte stores
constexpr uint32_t K1_F32_SBO = 16 * K1_F32_LBO;       // 8-row group stride (K = 64 tf32)
constexpr uint32_t K1_GA = 0;                          // tf32 [Kg'; Qg']: rows 128 x K = 64 channels
constexpr uint32_t K1_KD = K1_GA + 16 * K1_F32_SBO;    // tf32 Kd': rows 64 x K = 64 channels
constexpr uint32_t K1_GRAM_END = K1_KD + 8 * K1_F32_SBO;
// Kg'^T and V^T stay in shared memory, so their 8-row groups are padded by 16
// bytes: lanes whose rows d lie 8 apart then hit different banks and a warp
// stores one channel of its pairs at a time without conflicts.  Ke'^T keeps
// the record's layout (it is copied there as a whole).
constexpr uint32_t SBO_K64P = SBO_K64 + 16;
constexpr uint32_t K1_KGT = K1_GRAM_END;               // f16 Kg'^T: rows d (128) x K = i (64), SBO_K64P
constexpr uint32_t K1_VT = K1_KGT + 16 * SBO_K64P;     // f16 V^T  : rows e x K = i, SBO_K64P
constexpr uint32_t K1_KET = K1_VT + 16 * SBO_K64P;     // f16 Ke'^T: rows d x K = r
constexpr uint32_t K1_SMEM = K1_KET + 16384;
// later phases, inside [0, K1_GRAM_END)
constexpr int K1_P = 68;                 // fp32 row pitch of T (16-byte aligned rows)
constexpr int K1_PL = 68;                // fp32 row pitch of L (16-byte rows: conflict-free float4 stores by rows)
constexpr uint32_t K1_LM = 0;            // fp32 [64][68]  L (strict lower)
constexpr uint32_t K1_TM = 17408;        // fp32 [64][68]  T = (I + L)^-1
constexpr uint32_t K1_XS = 34816;        // fp32 [2][16][24] scratch of the 16 -> 32 merge
constexpr int K1_XSP = 24;               // its row pitch (conflict-free fragment loads)
constexpr uint32_t K1_MC = 37888;        // f16 Mc': rows r x K = i (64 x 64)
constexpr uint32_t K1_XW = 46080;        // fp32 [32][40] scratch of the 32 -> 64 merge
constexpr int K1_XWP = 40;               // its row pitch (conflict-free fragment loads)
constexpr uint32_t K1_TBK = 0;           // f16 T diag(beta rk): rows r x K = i, over L once T is built
constexpr uint32_t K1_TBV = 8192;        // f16 T diag(beta)
constexpr uint32_t K1_WKT = 0;           // f16 (diag(rk) Wk)^T: rows d x K = r, over TB once W is done
constexpr uint32_t K1_QG = K1_TM;        // f16 Qg': rows r of 128 channels, from registers over T
constexpr int K1_QGP = 136;              // its row pitch in f16 (272 bytes: conflict-free row reads by 16 lanes)
static_assert(K1_MC + 8192 <= K1_GRAM_END && K1_WKT + 16384 <= K1_MC, "later phases must fit the Gram region");
static_assert(K1_WKT + 16384 <= K1_QG && K1_QG + 64 * K1_QGP * 2 <= K1_XS, "Qg tile between Wk^T and the merge scratch");
static_assert(K1_LM + 64 * K1_PL * 4 <= K1_TM, "L below T");
static_assert(K1_TBV + 8192 <= K1_TM && K1_XS + 2 * 16 * K1_XSP * 4 <= K1_MC && K1_XW + 32 * K1_XWP * 4 <= K1_GRAM_END,
              "phase overlap");
static_assert(2 * (K1_SMEM + 8192) <= 228 * 1024, "two CTAs per SM");
constexpr int K1_THREADS = 256;
constexpr float kF16Max = 65504.f;       // largest finite f16
constexpr int kH32 = 32;                 // head count with its own K1 instance

// TMEM columns (256 allocated)
constexpr uint32_t T1_G = 0, T1_W1 = 64, T1_W2 = 128, T1_AP = 0, T1_QP = 128;

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint4 pack_f16x8(const float *x)
{
    return make_uint4(pack_f16x2(x[0], x[1]), pack_f16x2(x[2], x[3]), pack_f16x2(x[4], x[5]),
                      pack_f16x2(x[6], x[7]));
}

// The fused prologue's taps (kConv): fp32 [3 (q, k, v)][kConvTaps][128
// channels] after the kernel's other shared memory, the oldest taps zero for a
// narrower convolution.
constexpr uint32_t K1_TAPS_BYTES = 3 * kConvTaps * kD * 4;
// two CTAs per SM with the taps: dynamic + static (3 KB) + the 1 KB the SM reserves per CTA
static_assert(2 * (K1_SMEM + K1_TAPS_BYTES + 3072 + 1024) <= 228 * 1024, "two CTAs per SM with the taps");

// kConv: q, k, v pass through the short convolution as they are loaded.  kH > 0:
// the call has kH heads (row strides and head indices fold into constants).
template <bool kConv, int kH>
__global__ void __launch_bounds__(K1_THREADS, 2)
k1_tc_kernel(const bf16 *__restrict__ q, const bf16 *__restrict__ k, const bf16 *__restrict__ v,
             const float *__restrict__ g, const float *__restrict__ beta, int N, int H, SeqTable tab,
             uint8_t *__restrict__ ring, int seg_lo, int G, int slot_chunks, int slot, int scalar_gate,
             DevStatus *st, uint32_t wait_limit, const float *__restrict__ conv_w, int conv_width,
             int conv_silu, const bf16 *__restrict__ conv_in, int ahead, Bounds bd)
{
    if constexpr (kH > 0) H = kH;
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ uint64_t mbar, abar, dbar;
    __shared__ uint32_t tmem_sh;
    __shared__ __align__(16) float tot[8][64];   // per warp: totals of g over its 8 rows, per channel of the half
    // (16-byte aligned: read as float2 / float4)
    __shared__ __align__(16) float rq[kC];
    __shared__ __align__(16) float rk[kC];
    __shared__ __align__(16) float bs[kC];

    // grid: one CTA per (item, head), head fastest (CTAs running together read
    // adjacent 256-byte slices of the same token rows).  G == 0: the item is a
    // global chunk index and so is the record's.  G > 0: the item is (sequence
    // n, chunk seg_lo + i), i < G, and its record goes to position (n, i) of
    // ring slot `slot` (`slot_chunks` records per sequence).  Exits are uniform
    // and come before any allocation.
    const int h = (int)(blockIdx.x % (unsigned)H), item = (int)(blockIdx.x / (unsigned)H);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int n, lc, cu0, cu1;
    size_t ri;
    if (G == 0) {
        if (item >= tab.chunk_off[N]) return;
        n = find_seq_tc(tab.chunk_off, N, item);
        lc = item - tab.chunk_off[n];
        ri = (size_t)item;
        cu0 = tab.cu[n];
        cu1 = tab.cu[n + 1];
    } else {
        // n < N: both bounds of the sequence in one round trip, and its chunk
        // count follows from them (lc < ceil(len / C) exactly when lc C < len)
        n = item / G;
        lc = seg_lo + item % G;
        cu0 = tab.cu[n];
        cu1 = tab.cu[n + 1];
        if (lc * kC >= cu1 - cu0) return;
        ri = ((size_t)slot * N + n) * slot_chunks + item % G;
    }
    const int t0 = cu0 + lc * kC;
    // (debug build: rows past the token buffers' end count as rows past the
    // sequence's end, and a chunk with none left, or a record outside the
    // workspace, is skipped)
    const int L = dbg_rows(t0, min(kC, cu1 - t0), bd);
    if (kDebug && (L <= 0 || !dbg_in((int64_t)(ri * H + h), bd.records, kDbgRecord))) return;
    uint8_t *rec = ring + (ri * H + h) * REC_BYTES;
    // Qg' as an f16 operand tile (rows d, K = r; 16 KB) waits in registers
    // (each thread's two channels of its 8 rows, per channel half) until the
    // inverse is done and its shared-memory area is free
    uint32_t qgk[2][8];

    // 0. inputs of the first channel half.  Thread: rows rb .. rb + 7 of its
    //    warp, channels 64 p + 2 lane and + 1 of half p (4-byte bf16 pairs,
    //    8-byte gate pairs: each warp reads whole 128- and 256-byte row slices).
    const int rb = 8 * warp;
    const bf16 *qrow = q + ((size_t)t0 * H + h) * kD, *krow = k + ((size_t)t0 * H + h) * kD;
    const bf16 *vrow = v + ((size_t)t0 * H + h) * kD;
    size_t xstride = (size_t)H * kD;   // row stride of q, k, v (kConv: of their convolved copies)
    // q, k, v element pairs: read-only inputs, or (kConv) the convolved rows this
    // CTA wrote, which must not go through the read-only path
    // an element pair of q, k, v as fp32: bf16 inputs, or (kConv) f16 convolved rows
    auto up2 = [&](uint32_t u) -> float2 {
        if constexpr (kConv) {
            const __half2 h2 = *reinterpret_cast<const __half2 *>(&u);
            return __half22float2(h2);
        } else {
            return make_float2(bf_lo(u), bf_hi(u));
        }
    };
    auto ldx = [&](const bf16 *p) -> uint32_t {
        if constexpr (kConv) return *reinterpret_cast<const volatile uint32_t *>(p);
        else return __ldg(reinterpret_cast<const unsigned int *>(p));
    };
    // the gate: a decay per key channel ([T, H, Dk]) or one per row shared by
    // every channel ([T, H], then the same value fills both lanes of gv)
    const float *grow = g + ((size_t)t0 * H + h) * (scalar_gate ? 1 : kD);
    const size_t rstride = (size_t)H * kD;
    float2 gv[8];
    uint32_t qv[8], kv[8], vv[8];
    auto load_half = [&](int p) {
        int d = 64 * p + 2 * lane;
        asm volatile("" : "+r"(d));   // keeps the second half's loads after its barrier (registers)
        if (L == kC && !scalar_gate) {   // a full chunk with a per-channel gate: no row predicates
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const size_t o = (size_t)(rb + j) * rstride + d, ox = (size_t)(rb + j) * xstride + d;
                gv[j] = __ldg(reinterpret_cast<const float2 *>(grow + o));
                qv[j] = ldx(qrow + ox);
                kv[j] = ldx(krow + ox);
                vv[j] = ldx(vrow + ox);
            }
            return;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int r = rb + j;
            const bool valid = r < L;
            const size_t o = (size_t)r * rstride + d, ox = (size_t)r * xstride + d;
            if (scalar_gate) {
                const float gs = valid ? __ldg(grow + (size_t)r * H) : 0.f;
                gv[j] = make_float2(gs, gs);
            } else {
                gv[j] = valid ? __ldg(reinterpret_cast<const float2 *>(grow + o)) : make_float2(0.f, 0.f);
            }
            qv[j] = valid ? ldx(qrow + ox) : 0u;
            kv[j] = valid ? ldx(krow + ox) : 0u;
            vv[j] = valid ? ldx(vrow + ox) : 0u;
        }
    };
    if constexpr (kConv) {
        // The fused short convolution, as a first pass over the chunk: the taps
        // of this head into shared memory (zero on the older side of a narrower
        // convolution), then x'[r] = sum_i tap[i] x[r - 3 + i] in fp32 (x = 0
        // before the sequence's first token; x' = 0 from row L on), optionally
        // x' sigmoid(x'), rounded to f16 (11 significant bits; within the f16
        // range the operand tiles require of q, k, v anyway) into this chunk's
        // record, in areas the
        // record's own tiles fill only after the operand build (q' at the Q'
        // tile, k' at the Ke^T tile, v' at the Uv^T tile; rows of 128 channels).
        // The build below then reads q', k', v' from there.
        float *taps = reinterpret_cast<float *>(sm + K1_SMEM);
        for (int i = tid; i < 3 * kConvTaps * kD; i += K1_THREADS) {
            const int t = i / (kConvTaps * kD), j = (i / kD) % kConvTaps, c = i % kD;
            const int jw = j - (kConvTaps - conv_width);
            taps[i] = jw >= 0 ? __ldg(conv_w + (((size_t)t * conv_width + jw) * H + h) * kD + c) : 0.f;
        }
        __syncthreads();
        const int cp = 2 * (tid & 63), r0 = 16 * (tid >> 6);   // channel pair, 16 output rows
#pragma unroll 1
        for (int t = 0; t < 3; ++t) {
            const bf16 *src = t == 0 ? qrow : t == 1 ? krow : vrow;
            uint32_t *dst = reinterpret_cast<uint32_t *>(rec + (t == 0 ? REC_QP : t == 1 ? REC_KM : REC_UV));
            float2 w[kConvTaps], win[kConvTaps];
#pragma unroll
            for (int i = 0; i < kConvTaps; ++i) {
                w[i] = *reinterpret_cast<const float2 *>(taps + (t * kConvTaps + i) * kD + cp);
                // window slots 1 .. 3 start with rows r0 - 3 .. r0 - 1 (slot 0 is
                // shifted out before first use); each step shifts and appends a row.
                // Rows from L on feed only outputs that are zero and are not read
                // (in the sequence's last chunk they may lie past the buffers' end).
                const int rr = r0 - kConvTaps + i, pos = lc * kC + rr;   // position in the sequence
                uint32_t u = 0u;
                if (i > 0 && pos >= 0 && rr < L)
                    u = __ldg(reinterpret_cast<const unsigned int *>(src + (ptrdiff_t)rr * (ptrdiff_t)rstride + cp));
                else if (i > 0 && conv_in && pos >= -(conv_width - 1))   // the history before the sequence
                    u = __ldg(reinterpret_cast<const unsigned int *>(
                        conv_in + ((((size_t)n * 3 + t) * (conv_width - 1) + (conv_width - 1 + pos)) * H + h) * kD + cp));
                win[i] = make_float2(bf_lo(u), bf_hi(u));
            }
#pragma unroll 4
            for (int j = 0; j < 16; ++j) {
                const int r = r0 + j;
                const uint32_t u = r < L ? __ldg(reinterpret_cast<const unsigned int *>(src + (size_t)r * rstride + cp))
                                         : 0u;
#pragma unroll
                for (int i = 0; i < kConvTaps - 1; ++i) win[i] = win[i + 1];
                win[kConvTaps - 1] = make_float2(bf_lo(u), bf_hi(u));
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < kConvTaps; ++i) acc = __ffma2_rn(w[i], win[i], acc);
                if (conv_silu)
                    acc = make_float2(__fdividef(acc.x, 1.f + __expf(-acc.x)), __fdividef(acc.y, 1.f + __expf(-acc.y)));
                dst[(r * kD + cp) >> 1] = r < L ? pack_f16x2(acc.x, acc.y) : 0u;
            }
        }
        __syncthreads();   // the convolved rows are visible to the whole CTA (global memory)
        qrow = reinterpret_cast<const bf16 *>(rec + REC_QP);
        krow = reinterpret_cast<const bf16 *>(rec + REC_KM);
        vrow = reinterpret_cast<const bf16 *>(rec + REC_UV);
        xstride = kD;
    }
    const float beta_r = (tid < kC && tid < L) ? __ldg(beta + (size_t)(t0 + tid) * H + h) : 0.f;
    load_half(0);
    // L2 prefetch of the second channel half of this chunk's rows (one row
    // slice per thread: one 128-byte line of q, k or v, two of g), so that its
    // loads after the first half hit L2.  Line prefetches go through the
    // load/store path; the bulk prefetch of the same slices, issued through
    // the copy engine, held the issuing warps longer (calls 1.5% slower).
    {
        const int r = tid & 63, which = tid >> 6;   // q, k, v, g
        const char *base = which == 0 ? (const char *)q : which == 1 ? (const char *)k
                         : which == 2 ? (const char *)v : (const char *)g;
        const uint32_t esz = which == 3 ? 4u : 2u;
        if (!kConv && r < L && (which < 3 || !scalar_gate)) {
            const char *slice = base + (((size_t)(t0 + r) * H + h) * kD + 64) * esz;
            prefetch_line_l2(slice);
            if (esz == 4u) prefetch_line_l2(slice + 128);
        }
    }
    // ... and of the first half of the rows of the CTA `ahead` positions later
    // in the grid (segmented launches; `ahead` is half the SM count): that CTA
    // starts about half a wave later and then finds its first loads in L2,
    // instead of every CTA drawing its first 40 KB from HBM as it starts
    // (which, with the other CTAs doing the same, took about 1.8K cycles).
    // Prefetching a whole wave ahead, or both halves, measured slower.
    {
        const unsigned b2 = blockIdx.x + (unsigned)ahead;
        if (!kConv && G > 0 && ahead > 0 && b2 < gridDim.x) {
            const int h2 = (int)(b2 % (unsigned)H), item2 = (int)(b2 / (unsigned)H);
            const int n2 = item2 / G, lc2 = seg_lo + item2 % G;   // n2 < N (grid = N G H)
            const int c1 = tab.cu[n2 + 1], t02 = tab.cu[n2] + lc2 * kC;
            const int r = tid & 63, which = tid >> 6;   // q, k, v, g
            const char *base = which == 0 ? (const char *)q : which == 1 ? (const char *)k
                             : which == 2 ? (const char *)v : (const char *)g;
            const uint32_t esz = which == 3 ? 4u : 2u;
            if (t02 + r < c1 && (which < 3 || !scalar_gate) && dbg_in(t02 + r, bd.tokens, kDbgTokenRow)) {
                const char *slice = base + ((size_t)(t02 + r) * H + h2) * kD * esz;
                prefetch_line_l2(slice);
                if (esz == 4u) prefetch_line_l2(slice + 128);
            }
        }
    }

    if (warp == 0) {
        tmem_alloc(&tmem_sh, 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&mbar, 1);
        mbar_init(&abar, 1);
        mbar_init(&dbar, 1);
        fence_mbar_init();
    }
    // the TMEM address and the barriers are published by the loop's first CTA
    // barrier (the warps meanwhile compute their gate totals)
    uint32_t tm = 0;
    bool ok = true;
    bool strong = false;   // a decay factor of this thread's rows left the exact range
    // (debug build) The f16 operand tiles hold q, k and v before
    // normalisation: a q or k row of L2 norm 65504 or more (every element
    // beyond the f16 range, and some within it), or a v element beyond it, is
    // reported like a decay beyond range.  The release build leaves these
    // checks out (they measured 0.4-0.9% of a call).
    bool f16_over = false;
    float vmax = 0.f;
    float sqa[8];      // the first half's squared row norms after the exchange across lane bit 4

    // 1-3. per channel half p: cumulative gates, decayed operands, partial row
    //      norms; then the half's share of G' = [Kg'; Qg'] Kd'^T (tf32, M = 128,
    //      N = 64, K = 64: 8 instructions of K = 8, accumulating over the halves)
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const int d = 64 * p + 2 * lane;
        {
            float2 c = gv[0];
#pragma unroll
            for (int j = 1; j < 8; ++j) c = __fadd2_rn(c, gv[j]);
            *reinterpret_cast<float2 *>(&tot[warp][2 * lane]) = c;
        }
        if (p == 0 && tid < kC) bs[tid] = beta_r;
        if (p == 0) fence_before_sync();
        __syncthreads();
        if (p == 0) {
            fence_after_sync();
            tm = tmem_sh;
        }
        float2 pre = make_float2(0.f, 0.f), last = pre;   // totals of the warps before this one, of all
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            if (w == warp) pre = last;
            last = __fadd2_rn(last, *reinterpret_cast<const float2 *>(&tot[w][2 * lane]));
        }
        const float last0 = last.x, last1 = last.y;
        // Per channel the decays are referred to the midpoint B = b_last / 2 of
        // their range [b_last, 0]: the Gram factors e^(b - B) and e^(B - b) then
        // stay within e^(|b_last| / 2), and mu = e^B carries the rest
        // (Kg' = k e^(b - B) mu, Ke' = k e^(B - b) mu since b_last - B = B).
        const float2 ref = make_float2(0.5f * last0, 0.5f * last1);
        const float2 mu2 = make_float2(__expf(ref.x), __expf(ref.y));
        if (warp == 0) *reinterpret_cast<float2 *>(rec + REC_G + d * 4) = __fmul2_rn(mu2, mu2);
        uint32_t kg0[4], kg1[4], vf0[4], vf1[4], ke0[4], ke1[4], qp0[4], qp1[4];
        // this half's squared row norms: the exchange across lane bit 4 leaves q
        // of row rb + j (bit 4 clear) or k (set) in sq[j]; after the second half
        // the two halves' values are added and summed over the warp by halving
        // exchanges (bit 3 keeps four of the rows, and so on), so that lanes 2i
        // and 2i + 1 end with value i (q rows rb .. rb + 7, then k rows)
        float sq[8];
        const bool up16 = lane & 16;
        // byte offset of (row rb, channels 2 lane and + 1 of the half) in the tf32 K-major tiles
        const uint32_t gbase = kmaj_off4(rb, 2 * lane, K1_F32_LBO, K1_F32_SBO);
        // With g <= 0 each channel's b runs from 0 down to b_last, so |b - B| <=
        // |B|: while |B| <= kMaxDecayExp for every channel of the half (the
        // same channels in every warp), no factor can leave the range and the
        // clamps are skipped (a warp-uniform choice).
        const bool clamp = __any_sync(0xffffffffu, fabsf(ref.x) > kMaxDecayExp || fabsf(ref.y) > kMaxDecayExp);
        const float2 l2e2 = make_float2(kLog2e, kLog2e);
        const float2 refl2 = make_float2(-ref.x * kLog2e, -ref.y * kLog2e);
        auto build_rows = [&](auto kClamp) {
        float2 bb = pre;
#pragma unroll
        for (int j2 = 0; j2 < 8; j2 += 2) {
            float kgx[2][2], vx[2][2], kex[2][2], qgx[2][2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int j = j2 + u;
                bb = __fadd2_rn(bb, gv[j]);
                // e^(b - B) and e^(B - b) as 2^(+-(b - B) log2 e): one packed FMA for
                // the exponent, then the hardware base-2 exponential (flush to zero:
                // the factors stay at or above e^-80, far from the subnormal range)
                const float2 x = __ffma2_rn(bb, l2e2, refl2);
                float2 e, ei;
                if constexpr (decltype(kClamp)::value) {
                    strong |= fabsf(x.x) > kMaxDecayExp * kLog2e || fabsf(x.y) > kMaxDecayExp * kLog2e;
                    e = make_float2(ex2_ftz(fminf(x.x, kMaxDecayExp * kLog2e)), ex2_ftz(fminf(x.y, kMaxDecayExp * kLog2e)));
                    ei = make_float2(ex2_ftz(fminf(-x.x, kMaxDecayExp * kLog2e)), ex2_ftz(fminf(-x.y, kMaxDecayExp * kLog2e)));
                } else {
                    e = make_float2(ex2_ftz(x.x), ex2_ftz(x.y));
                    ei = make_float2(ex2_ftz(-x.x), ex2_ftz(-x.y));
                }
                const float2 qq = up2(qv[j]), kk = up2(kv[j]);
                // (kept row, row sent across lane bit 4) = (q, k), or (k, q) when the bit is set
                const float2 m0 = up16 ? make_float2(kk.x, qq.x) : make_float2(qq.x, kk.x);
                const float2 m1 = up16 ? make_float2(kk.y, qq.y) : make_float2(qq.y, kk.y);
                const float2 s2 = __ffma2_rn(m1, m1, __fmul2_rn(m0, m0));
                sq[j] = s2.x + __shfl_xor_sync(0xffffffffu, s2.y, 16);
                // Gram factors (referred to B), then the true decayed rows
                const float2 kgr = __fmul2_rn(kk, e), qgr = __fmul2_rn(qq, e), kd = __fmul2_rn(kk, ei);
                const float2 kg = __fmul2_rn(kgr, mu2), qg = __fmul2_rn(qgr, mu2);
                const float2 ke = __fmul2_rn(kd, mu2);   // k' e^(b_last - b)
                // row r = rb + j of the K-major tiles: the warp's 8-row group, then j
                uint8_t *const gp = sm + gbase + 16u * j;
                *reinterpret_cast<float2 *>(gp + K1_GA) = make_float2(round_tf32(kgr.x), round_tf32(kgr.y));
                *reinterpret_cast<float2 *>(gp + K1_GA + 8 * K1_F32_SBO) =   // row 64 + r
                    make_float2(round_tf32(qgr.x), round_tf32(qgr.y));
                *reinterpret_cast<float2 *>(gp + K1_KD) = make_float2(round_tf32(kd.x), round_tf32(kd.y));
                qgx[0][u] = qg.x; qgx[1][u] = qg.y;
                kgx[0][u] = kg.x; kgx[1][u] = kg.y;
                const float2 vf = up2(vv[j]);
                if constexpr (kDebug) vmax = fmaxf(vmax, fmaxf(fabsf(vf.x), fabsf(vf.y)));
                vx[0][u] = vf.x; vx[1][u] = vf.y;
                kex[0][u] = ke.x; kex[1][u] = ke.y;
            }
            qp0[j2 / 2] = pack_f16x2(qgx[0][0], qgx[0][1]);
            qp1[j2 / 2] = pack_f16x2(qgx[1][0], qgx[1][1]);
            kg0[j2 / 2] = pack_f16x2(kgx[0][0], kgx[0][1]);
            kg1[j2 / 2] = pack_f16x2(kgx[1][0], kgx[1][1]);
            vf0[j2 / 2] = pack_f16x2(vx[0][0], vx[0][1]);
            vf1[j2 / 2] = pack_f16x2(vx[1][0], vx[1][1]);
            ke0[j2 / 2] = pack_f16x2(kex[0][0], kex[0][1]);
            ke1[j2 / 2] = pack_f16x2(kex[1][0], kex[1][1]);
        }
        };
        // the Gram product of the previous half has read the tiles this half
        // overwrites (each thread waits itself; usually long done)
        if (p == 1) ok = ok && mbar_wait_bounded(&mbar, 0, wait_limit);
        if (clamp) build_rows(std::true_type{});
        else build_rows(std::false_type{});
        // The f16 operand tiles, the Qg' rows (kept in registers) and the norm
        // exchange, once the half's Gram product is issued: they overlap it (the
        // product reads only the tf32 tiles).
        auto finish_half = [&]() {
            // f16 operand rows d and d + 1, K = rows rb .. rb + 7: the padded tiles
            // row d, then row d + 1; in Ke'^T lanes 4-7 of each quarter-warp store
            // row d + 1 first, so that every store instruction covers eight distinct
            // rows modulo 8 (conflict-free either way).
            {
                const uint32_t pa = kmaj_off(d, rb, LBO_KIN, SBO_K64P), pb = kmaj_off(d + 1, rb, LBO_KIN, SBO_K64P);
                *reinterpret_cast<uint4 *>(sm + K1_KGT + pa) = make_uint4(kg0[0], kg0[1], kg0[2], kg0[3]);
                *reinterpret_cast<uint4 *>(sm + K1_KGT + pb) = make_uint4(kg1[0], kg1[1], kg1[2], kg1[3]);
                *reinterpret_cast<uint4 *>(sm + K1_VT + pa) = make_uint4(vf0[0], vf0[1], vf0[2], vf0[3]);
                *reinterpret_cast<uint4 *>(sm + K1_VT + pb) = make_uint4(vf1[0], vf1[1], vf1[2], vf1[3]);
                const bool sw = lane & 4;
                const uint32_t oa = kmaj_off(d + (sw ? 1 : 0), rb, LBO_KIN, SBO_K64);
                const uint32_t ob = kmaj_off(d + (sw ? 0 : 1), rb, LBO_KIN, SBO_K64);
                *reinterpret_cast<uint4 *>(sm + K1_KET + oa) =
                    sw ? make_uint4(ke1[0], ke1[1], ke1[2], ke1[3]) : make_uint4(ke0[0], ke0[1], ke0[2], ke0[3]);
                *reinterpret_cast<uint4 *>(sm + K1_KET + ob) =
                    sw ? make_uint4(ke0[0], ke0[1], ke0[2], ke0[3]) : make_uint4(ke1[0], ke1[1], ke1[2], ke1[3]);
            }
            // Qg'^T rows d and d + 1, kept in registers until phase 7
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                qgk[p][i] = qp0[i];
                qgk[p][4 + i] = qp1[i];
            }
            if (p == 0) {
#pragma unroll
                for (int j = 0; j < 8; ++j) sqa[j] = sq[j];
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) sq[j] += sqa[j];
#pragma unroll
                for (int w = 4; w >= 1; w >>= 1) {
                    const bool up = lane & (2 * w);
#pragma unroll
                    for (int i = 0; i < w; ++i) {
                        const float send = up ? sq[i] : sq[i + w], keep = up ? sq[i + w] : sq[i];
                        sq[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2 * w);
                    }
                }
                const float nsq = sq[0] + __shfl_xor_sync(0xffffffffu, sq[0], 1);   // row lane >> 1
                // the convolved rows (kConv) were written to the record by plain stores;
                // a bulk copy overwrites the k' rows after the inverse
                fence_async_global();
                if ((lane & 1) == 0) {
                    const int i = lane >> 1, r = rb + (i & 7);
                    (i < 8 ? rq : rk)[r] = r < L ? rsqrtf(nsq + 1e-6f) : 0.f;
                    if constexpr (kDebug) f16_over |= r < L && !(nsq < kF16Max * kF16Max);
                }
            }
        };
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (p == 0) load_half(1);          // next half's inputs in flight during the MMA
        if (tid == 0 && ok) {
            const uint32_t idesc = idesc_tf32(128, 64);
            const uint32_t a0 = smem_u32(sm + K1_GA), b0d = smem_u32(sm + K1_KD);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_tf32(tm + T1_G, make_desc(a0 + ks * 2 * K1_F32_LBO, K1_F32_LBO, K1_F32_SBO),
                         make_desc(b0d + ks * 2 * K1_F32_LBO, K1_F32_LBO, K1_F32_SBO), idesc, p > 0 || ks > 0);
            mma_commit(&mbar);
        }
        finish_half();
        fence_async_smem();   // the f16 tiles are read by later products
    }
    if (strong || f16_over || !(vmax < kF16Max)) record_status(st, (int32_t)KDA_ERR_UNSUPPORTED);
    __syncthreads();   // rq, rk and the f16 tiles of both halves are written
    ok = ok && mbar_wait_bounded(&mbar, 1, wait_limit);   // G' complete: the Gram region may be reused
    fence_after_sync();

    // 4. read G': lane quarter q4 = warp & 3 holds rows 32 q4 .. +31; warps w and
    //    w + 4 take columns [0, 32) and [32, 64).  Rows < 64: Kg' Kd'^T -> L;
    //    rows >= 64: Qg' Kd'^T -> Mc' (the row norm of q only).
    const int q4 = warp & 3, ch = warp >> 2;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    const int row = 32 * q4 + lane;
    float *Lm = reinterpret_cast<float *>(sm + K1_LM);
    float *Tm = reinterpret_cast<float *>(sm + K1_TM);
    float *Xs = reinterpret_cast<float *>(sm + K1_XS);
    float *Xw = reinterpret_cast<float *>(sm + K1_XW);
    if (ok && row < 64) {
        // L.  The inverse reads only its entries below the diagonal: they are
        // stored unmasked, and warp 4 (rows 0-31, columns 32-63, all on or above
        // the diagonal) neither reads G' nor stores.
        if (ch <= q4) {
            float gq[32];
            tmem_ld32(tm + lane_base + T1_G + 32 * ch, gq);
            tmem_ld_wait();
            const int r = row;
            const float sr = bs[r] * rk[r];
            const float2 sr2 = make_float2(sr, sr);
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const int col = 32 * ch + i;
                const float4 rk4 = *reinterpret_cast<const float4 *>(rk + col);
                const float2 l01 = __fmul2_rn(__fmul2_rn(sr2, make_float2(rk4.x, rk4.y)), make_float2(gq[i], gq[i + 1]));
                const float2 l23 =
                    __fmul2_rn(__fmul2_rn(sr2, make_float2(rk4.z, rk4.w)), make_float2(gq[i + 2], gq[i + 3]));
                *reinterpret_cast<float4 *>(Lm + r * K1_PL + col) = make_float4(l01.x, l01.y, l23.x, l23.y);
            }
        }
    } else if (ok) {
        // Mc' = rows r of G'_qk with the columns above the diagonal zeroed (K2
        // reads the whole tile).  Rows 32 dq .. + 31: columns 32 ch .. + 31 lie
        // wholly below the diagonal when ch < dq, wholly above it when ch > dq.
        const int r = row - 64, dq = q4 - 2;
        auto store_mc = [&](auto kMode) {   // 0: masked, 1: below, 2: above
            constexpr int mode = decltype(kMode)::value;
            float gq[32];
            if constexpr (mode != 2) {
                tmem_ld32(tm + lane_base + T1_G + 32 * ch, gq);
                tmem_ld_wait();
            }
            const float sr = rq[r];
#pragma unroll
            for (int i8 = 0; i8 < 32; i8 += 8) {
                float m8[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if constexpr (mode == 0) m8[j] = (32 * ch + i8 + j <= r) ? sr * gq[i8 + j] : 0.f;
                    else if constexpr (mode == 1) m8[j] = sr * gq[i8 + j];
                    else m8[j] = 0.f;
                }
                *reinterpret_cast<uint4 *>(sm + K1_MC + kmaj_off(r, 32 * ch + i8, LBO_KIN, SBO_K64)) = pack_f16x8(m8);
            }
        };
        if (ch == dq) store_mc(std::integral_constant<int, 0>{});
        else if (ch < dq) store_mc(std::integral_constant<int, 1>{});
        else store_mc(std::integral_constant<int, 2>{});
    }
    fence_async_smem();
    __syncthreads();
    // Ke'^T and Mc', already K2's operand tiles, go to the record by bulk copies
    // while the inverse runs (waited for before the CTA exits; neither tile is
    // overwritten)
    if (tid == 0) {
        static_assert(REC_MC == REC_KM + 16384, "Mc follows Ke^T");
        bulk_s2g(rec + REC_KM, sm + K1_KET, 16384);
        bulk_s2g(rec + REC_MC, sm + K1_MC, 8192);
        bulk_commit();
    }
    // 5. T = (I + L)^-1.  Diagonal 16 x 16 blocks by forward substitution (one
    //    column per thread), then two doubling merges, 16 -> 32 and 32 -> 64:
    //    for a lower block pair A (top) and B, T_BA = -T_BB (L_BA T_AA).
    if (tid < 64) {
        // column c of block blk, right-looking: once entry rr is final it is
        // taken out of every later row at once, so the dependent chain is one
        // FMA per row (entries above the diagonal stay zero: they start at
        // zero and only ever subtract multiples of zeros)
        const int blk = tid >> 4, c = tid & 15, col = 16 * blk + c;
        const float *lb = Lm + 16 * blk * (K1_PL + 1);   // L block blk, row stride K1_PL
        float x[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = (j == c) ? 1.f : 0.f;
#pragma unroll
        for (int rr = 0; rr < 15; ++rr)
#pragma unroll
            for (int j = rr + 1; j < 16; ++j) x[j] = fmaf(-lb[j * K1_PL + rr], x[rr], x[j]);
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) Tm[(16 * blk + rr) * K1_P + col] = x[rr];
    } else if (tid < 192) {
        // zeros in the 16 x 16 blocks above the diagonal of T_AA and T_BB
        // (rows 0-15 x columns 16-31, rows 32-47 x columns 48-63): the merges
        // below then run over whole blocks, without triangular bounds
        const int z = tid - 64, r = (z >> 2) + (z >= 64 ? 16 : 0), c4 = 16 + 4 * (z & 3) + (z >= 64 ? 32 : 0);
        *reinterpret_cast<float4 *>(Tm + r * K1_P + c4) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    if (warp < 4) {
        // 16 -> 32 on the warp-level tensor-core path: warp w takes pair k = w >> 1
        // (A = block 2k, B = block 2k + 1) and the 16 x 8 tile of columns
        // 8 (w & 1) of the pair's 16.  Each warp reads back only its own tile
        // of X, so a warp barrier separates the two products.
        const int g = lane >> 2, t = lane & 3, k2 = warp >> 1, n0 = 8 * (warp & 1);
        const int a0 = 32 * k2, b0 = a0 + 16;
        float *xs = Xs + k2 * 16 * K1_XSP;
        {   // X = L_BA T_AA (T_AA[k][n] = 0 for k < n: k starts at n0)
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            const float *la = Lm + (b0 + g) * K1_PL + a0 + t;
#pragma unroll
            for (int k0 = 0; k0 < 16; k0 += 8) {
                if (k0 < n0) continue;
                const float a[4] = {la[k0], la[8 * K1_PL + k0], la[k0 + 4], la[8 * K1_PL + k0 + 4]};
                const float b[2] = {Tm[(a0 + k0 + t) * K1_P + a0 + n0 + g], Tm[(a0 + k0 + t + 4) * K1_P + a0 + n0 + g]};
                mma_tf32x3(d, a, b);
            }
            *reinterpret_cast<float2 *>(xs + g * K1_XSP + n0 + 2 * t) = make_float2(d[0], d[1]);
            *reinterpret_cast<float2 *>(xs + (g + 8) * K1_XSP + n0 + 2 * t) = make_float2(d[2], d[3]);
        }
        __syncwarp();
        {   // T_BA = -T_BB X (T_BB unit lower triangular, zeros above its diagonal)
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            const float *ta = Tm + (b0 + g) * K1_P + b0 + t;
#pragma unroll
            for (int k0 = 0; k0 < 16; k0 += 8) {
                const float a[4] = {ta[k0], ta[8 * K1_P + k0], ta[k0 + 4], ta[8 * K1_P + k0 + 4]};
                const float b[2] = {xs[(k0 + t) * K1_XSP + n0 + g], xs[(k0 + t + 4) * K1_XSP + n0 + g]};
                mma_tf32x3(d, a, b);
            }
            *reinterpret_cast<float2 *>(Tm + (b0 + g) * K1_P + a0 + n0 + 2 * t) = make_float2(-d[0], -d[1]);
            *reinterpret_cast<float2 *>(Tm + (b0 + g + 8) * K1_P + a0 + n0 + 2 * t) = make_float2(-d[2], -d[3]);
        }
    }
    __syncthreads();
    {   // 32 -> 64 (A = rows 0-31, B = rows 32-63) on the warp-level tensor-core
        // path: warp w takes the 16 x 8 output tile at rows 16 (w & 1), columns
        // 8 (w >> 1), over K = 32 in steps of 8 (mma_tf32x3).  Steps whose
        // operand block lies above a triangular factor's diagonal are zero and
        // skipped (a warp-uniform bound).
        const int g = lane >> 2, t = lane & 3, m0 = 16 * (warp & 1), n0 = 8 * (warp >> 1);
        {   // X = L_BA T_AA: T_AA[k][n] = 0 for k < n, so k starts at n0
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            const float *la = Lm + (32 + m0 + g) * K1_PL + t;
#pragma unroll
            for (int k0 = 0; k0 < 32; k0 += 8) {
                if (k0 < n0) continue;
                const float a[4] = {la[k0], la[8 * K1_PL + k0], la[k0 + 4], la[8 * K1_PL + k0 + 4]};
                const float b[2] = {Tm[(k0 + t) * K1_P + n0 + g], Tm[(k0 + t + 4) * K1_P + n0 + g]};
                mma_tf32x3(d, a, b);
            }
            *reinterpret_cast<float2 *>(Xw + (m0 + g) * K1_XWP + n0 + 2 * t) = make_float2(d[0], d[1]);
            *reinterpret_cast<float2 *>(Xw + (m0 + g + 8) * K1_XWP + n0 + 2 * t) = make_float2(d[2], d[3]);
        }
        __syncthreads();
        // T_BA = -T_BB X (T_BB[m][k] = 0 for k > m, so k stays below m0 + 16).
        // The entries go straight into the f16 operands T diag(beta rk) and
        // T diag(beta) (rows r, K = i), which overwrite L.
        {
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            const float *ta = Tm + (32 + m0 + g) * K1_P + 32 + t;
#pragma unroll
            for (int k0 = 0; k0 < 32; k0 += 8) {
                if (k0 >= m0 + 16) continue;
                const float a[4] = {ta[k0], ta[8 * K1_P + k0], ta[k0 + 4], ta[8 * K1_P + k0 + 4]};
                const float b[2] = {Xw[(k0 + t) * K1_XWP + n0 + g], Xw[(k0 + t + 4) * K1_XWP + n0 + g]};
                mma_tf32x3(d, a, b);
            }
            const int c = n0 + 2 * t;
            const float2 b2 = *reinterpret_cast<const float2 *>(bs + c);
            const float2 k2 = *reinterpret_cast<const float2 *>(rk + c);
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {
                const float2 v = __fmul2_rn(make_float2(-d[2 * h8], -d[2 * h8 + 1]), b2);
                const float2 kv = __fmul2_rn(v, k2);
                const uint32_t o = kmaj_off(32 + m0 + g + 8 * h8, c, LBO_KIN, SBO_K64);
                *reinterpret_cast<uint32_t *>(sm + K1_TBK + o) = pack_f16x2(kv.x, kv.y);
                *reinterpret_cast<uint32_t *>(sm + K1_TBV + o) = pack_f16x2(v.x, v.y);
            }
        }
        // 6. the other blocks of T (T_AA, T_BB, final since the 16 -> 32 merge,
        //    and the zeros above the diagonal) -> the same operands, in pieces
        //    of 8 columns (warp = column piece, lane = row): thread t < 128 takes
        //    rows 0-31 x column pieces 0-3 (T_AA) and stores the zero pieces 4-7
        //    of the same rows, thread t >= 128 rows 32-63 x column pieces 4-7 (T_BB)
        if (tid < 128) {
            const uint32_t o = kmaj_off(tid & 31, 8 * (4 + (tid >> 5)), LBO_KIN, SBO_K64);
            *reinterpret_cast<uint4 *>(sm + K1_TBK + o) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(sm + K1_TBV + o) = make_uint4(0u, 0u, 0u, 0u);
        }
        static_assert(K1_THREADS == 256, "one T piece per thread");
        {
            const int r = (tid < 128 ? 0 : 32) + (tid & 31), c0 = 8 * (tid >> 5);
            float tk[8], tv[8];
#pragma unroll
            for (int j4 = 0; j4 < 8; j4 += 4) {
                const int ib = c0 + j4;
                const float4 t4 = *reinterpret_cast<const float4 *>(Tm + r * K1_P + ib);
                const float4 b4 = *reinterpret_cast<const float4 *>(bs + ib);
                const float4 k4 = *reinterpret_cast<const float4 *>(rk + ib);
                const float2 v01 = __fmul2_rn(make_float2(t4.x, t4.y), make_float2(b4.x, b4.y));
                const float2 v23 = __fmul2_rn(make_float2(t4.z, t4.w), make_float2(b4.z, b4.w));
                const float2 k01 = __fmul2_rn(v01, make_float2(k4.x, k4.y));
                const float2 k23 = __fmul2_rn(v23, make_float2(k4.z, k4.w));
                const float vv4[4] = {v01.x, v01.y, v23.x, v23.y}, kk4[4] = {k01.x, k01.y, k23.x, k23.y};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const bool in = ib + u <= r;   // T is lower triangular; above it lies stale data
                    tv[j4 + u] = in ? vv4[u] : 0.f;
                    tk[j4 + u] = in ? kk4[u] : 0.f;
                }
            }
            const uint32_t o = kmaj_off(r, c0, LBO_KIN, SBO_K64);
            *reinterpret_cast<uint4 *>(sm + K1_TBK + o) = pack_f16x8(tk);
            *reinterpret_cast<uint4 *>(sm + K1_TBV + o) = pack_f16x8(tv);
        }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // 7. Wk^T = Kg'^T (T diag(beta rk))^T and Uv^T = V^T (T diag beta)^T  (M = 128, N = 64, K = 64)
    if (tid == 0 && ok) {
        const uint32_t idesc = idesc_f16(128, 64);
        const uint32_t akg = smem_u32(sm + K1_KGT), av = smem_u32(sm + K1_VT);
        const uint32_t btk = smem_u32(sm + K1_TBK), btv = smem_u32(sm + K1_TBV);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            mma_f16(tm + T1_W1, make_desc(akg + ks * 256, LBO_KIN, SBO_K64P),
                    make_desc(btk + ks * 256, LBO_KIN, SBO_K64), idesc, ks > 0);
            mma_f16(tm + T1_W2, make_desc(av + ks * 256, LBO_KIN, SBO_K64P),
                    make_desc(btv + ks * 256, LBO_KIN, SBO_K64), idesc, ks > 0);
        }
        mma_commit(&mbar);
    }
    // Qg' from registers into shared memory over T, free now that the inverse
    // is done (after the W product is issued): plain rows (r, 128 channels of
    // f16), read back by the Q' readout (each register pair holds rows 2i and
    // 2i + 1 of channels d and d + 1)
#pragma unroll
    for (int p = 0; p < 2; ++p)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t *qrow = reinterpret_cast<uint32_t *>(sm + K1_QG) + (size_t)(rb + 2 * i) * (K1_QGP / 2) + 32 * p + lane;
            qrow[0] = __byte_perm(qgk[p][i], qgk[p][4 + i], 0x5410);
            qrow[K1_QGP / 2] = __byte_perm(qgk[p][i], qgk[p][4 + i], 0x7632);
        }
    // From here on each thread waits for the products itself (all lanes of a
    // warp poll together): what follows each wait reads only TMEM and writes
    // areas no other warp still reads, so no CTA barrier is needed there.
    ok = ok && mbar_wait_bounded(&mbar, 0, wait_limit);
    fence_after_sync();

    // 8. (-diag(rk) Wk)^T -> smem operand (rows d, K = r); Uv^T stays in
    //    registers until the products of phase 9 are issued.  Warp w reads
    //    lanes of quarter q4, columns [32 ch, 32 ch + 32).
    float wu[4][16];   // Wk^T and Uv^T, columns c and c + 16: all four loads before one wait
    if (ok) {
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
            tmem_ld16(tm + lane_base + T1_W1 + 32 * ch + 16 * c2, wu[2 * c2]);
            tmem_ld16(tm + lane_base + T1_W2 + 32 * ch + 16 * c2, wu[2 * c2 + 1]);
        }
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; c += 16) {
            float (&w)[16] = wu[c / 8];
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                const float2 s2 = *reinterpret_cast<const float2 *>(rk + 32 * ch + c + j);
                // Wk's tile carries -rk: the products of phase 9 come out as A'
                // and -Mc Wk directly
                const float2 w2 = __fmul2_rn(make_float2(w[j], w[j + 1]), make_float2(-s2.x, -s2.y));
                w[j] = w2.x; w[j + 1] = w2.y;
            }
#pragma unroll
            for (int h8 = 0; h8 < 16; h8 += 8)
                *reinterpret_cast<uint4 *>(sm + K1_WKT + kmaj_off(row, 32 * ch + c + h8, LBO_KIN, SBO_K64)) =
                    pack_f16x8(w + h8);
        }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // 9. A' = -Ke'^T diag(rk) Wk (M = 128, N = 128, K = 64), committed on its own so
    //    that its readout overlaps the second product; -Mc Wk = -Mc' diag(rk) Wk
    //    (M = 64, N = 128, K = 64), to which the Q' readout adds diag(rq) Qg'
    if (tid == 0 && ok) {
        const uint32_t ake = smem_u32(sm + K1_KET), amc = smem_u32(sm + K1_MC), bw = smem_u32(sm + K1_WKT);
        const uint32_t id128 = idesc_f16(128, 128), id64 = idesc_f16(64, 128);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_f16(tm + T1_AP, make_desc(ake + ks * 256, LBO_KIN, SBO_K64),
                    make_desc(bw + ks * 256, LBO_KIN, SBO_K64), id128, ks > 0);
        mma_commit(&abar);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_f16(tm + T1_QP, make_desc(amc + ks * 256, LBO_KIN, SBO_K64),
                    make_desc(bw + ks * 256, LBO_KIN, SBO_K64), id64, ks > 0);
        mma_commit(&mbar);
    }
    // (diag(rk) Uv)^T -> record (rows e, K = r) while the products run
    if (ok) {
#pragma unroll
        for (int c = 0; c < 32; c += 16) {
            float (&u)[16] = wu[c / 8 + 1];
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                const float2 s2 = *reinterpret_cast<const float2 *>(rk + 32 * ch + c + j);
                const float2 u2 = __fmul2_rn(make_float2(u[j], u[j + 1]), s2);
                u[j] = u2.x; u[j + 1] = u2.y;
            }
#pragma unroll
            for (int h8 = 0; h8 < 16; h8 += 8)
                *reinterpret_cast<uint4 *>(rec + REC_UV + kmaj_off(row, 32 * ch + c + h8, LBO_KIN, SBO_K64)) =
                    pack_f16x8(u + h8);
        }
    }
    ok = ok && mbar_wait_bounded(&abar, 0, wait_limit);
    fence_after_sync();

    // 10. A' -> record (rows d, K = d'); columns [64 ch, 64 ch + 64), all four
    //     16-column loads in flight before one wait
    if (ok) {
        float a[4][16];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld16(tm + lane_base + T1_AP + 64 * ch + 16 * q, a[q]);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int h8 = 0; h8 < 16; h8 += 8)
                *reinterpret_cast<uint4 *>(rec + REC_AP + kmaj_off(row, 64 * ch + 16 * q + h8, LBO_KIN, SBO_K128)) =
                    pack_f16x8(a[q] + h8);
    }
    ok = ok && mbar_wait_bounded(&mbar, 1, wait_limit);
    fence_after_sync();
    // 11. Q' = diag(rq) Qg' - Mc Wk -> record: the M = 64 accumulator puts row
    //     r = 16 q4 + l in lane 32 q4 + l (l < 16); the readout adds rq[r] Qg'[r]
    //     (fp32) from the plain rows of Qg' in shared memory
    if (ok) {
        const int r = 16 * q4 + lane;
        float a[4][16];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld16(tm + lane_base + T1_QP + 64 * ch + 16 * q, a[q]);
        tmem_ld_wait();
        if (lane < 16) {
            const float rqr = rq[r];
            const uint4 *qg = reinterpret_cast<const uint4 *>(sm + K1_QG + (size_t)r * K1_QGP * 2 + 64 * ch * 2);
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int h8 = 0; h8 < 16; h8 += 8) {
                    const uint4 g8 = qg[(16 * q + h8) / 8];
                    const uint32_t gw[4] = {g8.x, g8.y, g8.z, g8.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float2 gf = __half22float2(*reinterpret_cast<const __half2 *>(&gw[j]));
                        a[q][h8 + 2 * j] = fmaf(rqr, gf.x, a[q][h8 + 2 * j]);
                        a[q][h8 + 2 * j + 1] = fmaf(rqr, gf.y, a[q][h8 + 2 * j + 1]);
                    }
                    *reinterpret_cast<uint4 *>(rec + REC_QP + kmaj_off(r, 64 * ch + 16 * q + h8, LBO_KIN, SBO_K128)) =
                        pack_f16x8(a[q] + h8);
                }
        }
    }
    if (!ok && lane == 0) record_timeout(st);   // any warp whose wait gave up
    if (!ok && tid == 0) {
        // A wait of the issuing thread gave up: before the TMEM is freed and the
        // shared memory handed back, every MMA it issued must have completed (a
        // commit arrives once all earlier MMAs are done).
        mma_commit(&dbar);
        mbar_wait_bounded(&dbar, 0, kDrainLimit);
    }
    if (tid == 0) bulk_wait_all();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tm, 256);
}

// ============================================================ K2
// One CTA per (sequence, head), serial over the sequence's chunks.
//   16 state warps: thread (e = 32 (w & 3) + lane, quarter qd = w >> 2) keeps
//   S[d][e] for d in [32 qd, 32 qd + 32) in fp32 registers and writes output
//   rows [16 qd, 16 qd + 16) of column e; one thread of a 17th warp issues the
//   MMAs and one of an 18th the record copies into a 2-stage ring.
// Per chunk one product [A' S | Q' S]^T (N = 192: the record keeps the A'
// and Q' tiles adjacent) accumulates over the eight K steps of d', issued in
// one run once the state threads have written all of S^T.  S^T, the
// product's A operand, lives in TMEM (f16, row e in lane e): the state threads
// hand it on with tcgen05.st instead of shared-memory stores and a proxy
// fence, and the tensor core reads only the B operand from shared memory.
// The state threads read P, hand the next S^T on, then read O, so the next
// chunk's product overwrites them while this chunk's output is written to
// memory.
constexpr int K2_STAGES = 2;
constexpr int kGamSlots = 4;  // gamma vectors kept apart from the stages (ring of 4)
constexpr uint32_t K2_GAM = K2_STAGES * REC_BYTES;     // fp32 gamma [kGamSlots][128]
constexpr int K2_STATE_WARPS = 16;
// per state warp a 1 KB tile that turns its 16 output rows of 32 columns into
// 16-byte pieces of rows
constexpr uint32_t K2_OST = K2_GAM + kGamSlots * 512;
constexpr uint32_t K2_SMEM = K2_OST + K2_STATE_WARPS * 1024;
constexpr int K2_STATE_THREADS = 32 * K2_STATE_WARPS;
constexpr int K2_THREADS = K2_STATE_THREADS + 64;   // + the MMA issuer's warp and the copy warp
static_assert(K2_SMEM <= 227 * 1024 - 1024, "shared memory");
// TMEM columns (512 allocated): accumulator buffer b at 256 b, (A' S)^T in its
// columns 0-127 and (Q' S)^T in 128-191; S^T in f16 at 192-255 (row e in lane
// e, d and d + 1 in one column)
constexpr uint32_t T2_P = 0, T2_O = 128, T2_S = 192;

// This thread's 32 rows d of S^T (lane e, columns T2_S + 16 qd ..) in f16,
// stored and complete when the function returns.
__device__ __forceinline__ void write_state_tmem(uint32_t taddr, const float (&S)[32])
{
    float pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = __uint_as_float(pack_f16x2(S[2 * i], S[2 * i + 1]));
    tmem_st16(taddr, pk);
    tmem_st_wait();
}


// kMulti false: one chain per CTA (grid = chains); true: chains in turn.
// kGate: the output is o * sigmoid(gate) (the fused epilogue), gate [T, H, Dv] bf16.
template <bool kMulti, bool kGate>
__global__ void __maxnreg__(96)   // 18 warps: at most 5 per SM sub-partition x 32 x 96 <= 16384
k2_tc_kernel(StateIO io, int N, int H, SeqTable tab,
             const uint8_t *__restrict__ ring, int seg_lo, int G, int slot_chunks, int slot,
             float *__restrict__ carry, bf16 *__restrict__ out, DevStatus *st, uint32_t wait_limit,
             const bf16 *__restrict__ gate, Bounds bd)
{
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ uint64_t full[K2_STAGES], fullr[K2_STAGES], empty[K2_STAGES], emptyr[K2_STAGES], gfull[kGamSlots],
        sdone, pread[2], sready, dbar;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // A CTA runs the chains (sequence n, head h) = blockIdx.x, blockIdx.x +
    // gridDim.x, ... one after another (one chain per CTA when the grid covers
    // them all; fewer, longer-lived CTAs leave the other SMs to K1).  Barrier
    // phases and ring positions follow one chunk count that runs on across the
    // CTA's chains: the chain's local chunk c is chunk base + c of the CTA.
    if (tid == 0) {
        for (int s = 0; s < K2_STAGES; ++s) {
            mbar_init(&full[s], 1);     // [A'; Q'] of the stage landed
            mbar_init(&fullr[s], 1);    // [Ke^T; Mc], Uv^T of the stage landed
            mbar_init(&empty[s], 1);    // the MMA's commits: the stage's parts were read (the state
            mbar_init(&emptyr[s], 1);   // threads read gamma from its own ring)
        }
        for (int j = 0; j < kGamSlots; ++j) mbar_init(&gfull[j], 1);
        mbar_init(&sdone, 1);
        mbar_init(&dbar, 1);
        for (int j = 0; j < 2; ++j) mbar_init(&pread[j], K2_STATE_THREADS);   // per accumulator buffer
        mbar_init(&sready, K2_STATE_THREADS);   // S^T of the next chunk written
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

    const int q4 = warp & 3, qd = warp >> 2;
    const int e = 32 * q4 + lane;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    // Lane 0 of the warp after the state warps issues the MMAs, lane 0 of the
    // last warp the record copies (an MMA issue holds its thread for about the
    // pipe's time per step, so copies issued by the same thread would wait
    // behind the products); the other lanes of those warps have no part.
    const bool issuer = tid == K2_STATE_THREADS;
    const bool copier = tid == K2_STATE_THREADS + 32;
    const bool state_thread = tid < K2_STATE_THREADS;
    constexpr size_t DD = (size_t)kD * kD;
    const int stride = io.stride;
    int copied = 0;          // (copier) chunks whose second record part was issued, CTA count
    int copied_r = 0;        // (copier) ... whose first part and gamma were issued
    int base_run = 0;        // chunks of this CTA's earlier chains
    bool alive = true;

    for (int chain = blockIdx.x; chain < N * H && alive && (issuer || copier || state_thread); chain += gridDim.x) {
        const int base = kMulti ? base_run : 0;
        const int n = chain / H, h = chain % H;
        // This launch covers the sequence's local chunks [c_lo, c_lo + nch) of
        // segment [seg_lo, seg_lo + G); the state enters from the initial state
        // (first segment) or the carry buffer and leaves to the final state
        // (last segment) or the carry.  G == 0: the whole sequence, records
        // indexed by global chunk.
        const int nch_seq = tab.chunk_off[n + 1] - tab.chunk_off[n];
        const int c_lo = G == 0 ? 0 : seg_lo;
        const int nch = G == 0 ? nch_seq : max(0, min(seg_lo + G, nch_seq) - seg_lo);
        const int seq_t0 = tab.cu[n], seq_t1 = tab.cu[n + 1];
        const bool first_seg = c_lo == 0, last_seg = G == 0 || seg_lo + G >= nch_seq;
        const size_t sbase = ((size_t)n * H + h) * DD;   // this chain's block of the carry buffer
        // initial and final state blocks of this chain (dense arrays or pool
        // slots), looked up where they are used so that nothing of them stays
        // live across the chunk loop
        auto init_block = [&]() -> const float * {
            const int64_t is = io.init ? pool_slot(io.init_slots, n, io.pool) : -1;
            return is >= 0 && dbg_in(is, bd.states, kDbgState) ? io.init + ((size_t)is * H + h) * DD : nullptr;
        };
        auto final_block = [&]() -> float * {
            const int64_t fs = io.fin ? pool_slot(io.final_slots, n, io.pool) : -1;
            return fs >= 0 && dbg_in(fs, bd.states, kDbgState) ? io.fin + ((size_t)fs * H + h) * DD : nullptr;
        };
        const size_t rec_base = G == 0 ? (size_t)tab.chunk_off[n] : ((size_t)slot * N + n) * slot_chunks;
        if (nch == 0) {   // nothing of this sequence here; an empty sequence keeps its state
            if (state_thread && first_seg && nch_seq == 0)
                if (float *fin_blk = final_block()) {
                    const float *init_blk = init_block();
                    for (int i = tid; i < kD * kD; i += K2_STATE_THREADS) fin_blk[i] = init_blk ? init_blk[i] : 0.f;
                }
            continue;
        }
        // record of the sequence's chunk c_lo + i
        auto rec_at = [&](int i) { return ring + ((rec_base + i) * H + h) * REC_BYTES; };

        if (copier) {
            // ---------------------------------------------------------- copies
            // Record of local chunk c -> stage cc % K2_STAGES (cc = base + c), in
            // two parts with barriers of their own: the tiles of the
            // state-independent steps (Ke^T, Mc, Uv^T; 40 KB), once those steps
            // of chunk cc - K2_STAGES have read the stage's copy, and [A'; Q']
            // (48 KB), once that chunk's product is complete.  The first part's
            // stage frees up about a chunk earlier, so two parts are in flight
            // most of the time; gamma goes into its own slot with its own barrier
            // (the state threads read it later).
            static_assert(REC_KM + 40960 == REC_G && REC_AP == 0, "record parts");
            // (debug build) the chain's records lie inside the workspace, else
            // nothing is copied and the CTA's other roles are told to stop
            if (!dbg_in((int64_t)((rec_base + nch - 1) * H + h), bd.records, kDbgRecord)) {
                *abort_v = 1;
                alive = false;
            }
            for (int c = 0; c < nch && alive; ++c) {
                const int cc = base + c, s = cc % K2_STAGES;
                if (cc >= K2_STAGES &&
                    !wait_or_abort(&emptyr[s], ((cc - K2_STAGES) / K2_STAGES) & 1, abort_v, wait_limit)) {
                    alive = false;
                    break;
                }
                mbar_arrive_expect_tx(&fullr[s], REC_G - REC_KM);
                bulk_g2s(sm + s * REC_BYTES + REC_KM, rec_at(c) + REC_KM, REC_G - REC_KM, &fullr[s]);
                mbar_arrive_expect_tx(&gfull[cc % kGamSlots], 512);
                bulk_g2s(sm + K2_GAM + (cc % kGamSlots) * 512, rec_at(c) + REC_G, 512, &gfull[cc % kGamSlots]);
                copied_r = cc + 1;
                if (cc >= K2_STAGES &&
                    !wait_or_abort(&empty[s], ((cc - K2_STAGES) / K2_STAGES) & 1, abort_v, wait_limit)) {
                    alive = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], REC_KM);
                bulk_g2s(sm + s * REC_BYTES, rec_at(c), REC_KM, &full[s]);
                copied = cc + 1;
            }
        } else if (issuer) {
            // chunk cc: D = [P | O], P = (A' S + Ke^T Uv)^T, O = (Q' S + Mc Uv)^T,
            // in TMEM buffer cc & 1 (N = 192 rows of B: d, then r).  The K = r
            // steps (A = Uv^T) do not involve the state: they are issued as soon
            // as their part of the record has landed and the buffer's previous
            // contents (chunk cc - 2) were read, so they run while the state
            // threads still work on chunk cc - 1; the K = d' steps (A = S^T)
            // follow once the state threads have written S^T.
            auto issue_rpart = [&](int cc) -> bool {
                const int s = cc % K2_STAGES;
                const uint32_t stg = smem_u32(sm + s * REC_BYTES), acc = tm + T2_P + 256 * (cc & 1);
                const uint32_t idesc = idesc_f16(128, 192);
                bool okw = wait_or_abort(&fullr[s], (cc / K2_STAGES) & 1, abort_v, wait_limit);
                okw = okw && (cc < 2 || wait_or_abort(&pread[cc & 1], ((cc >> 1) - 1) & 1, abort_v, wait_limit));
                if (!okw) return false;
                fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_f16(acc, make_desc(stg + REC_UV + ks * 256, LBO_KIN, SBO_K64),
                            make_desc(stg + REC_KM + ks * 256, LBO_KIN, SBO_K64), idesc, ks > 0);
                mma_commit(&emptyr[s]);
                return true;
            };
            auto issue_dpart = [&](int cc) -> bool {
                const int s = cc % K2_STAGES;
                const uint32_t stg = smem_u32(sm + s * REC_BYTES), acc = tm + T2_P + 256 * (cc & 1);
                const uint32_t sop = tm + T2_S;   // S^T in TMEM: a K step of 16 is 8 columns
                const uint32_t idesc = idesc_f16(128, 192);
                // all of S^T, then the eight steps in one run: issuing them half by
                // half as each half of S^T arrived measured 0.5-1.4% slower, and by
                // quarters 2-6% slower (a wait between MMA issues costs more than
                // the earlier start gains)
                if (!wait_or_abort(&full[s], (cc / K2_STAGES) & 1, abort_v, wait_limit) ||
                    !wait_or_abort(&sready, cc & 1, abort_v, wait_limit))
                    return false;
                fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_f16_ts(acc, sop + 8 * ks, make_desc(stg + REC_AP + ks * 256, LBO_KIN, SBO_K128), idesc, 1);
                mma_commit(&sdone);
                mma_commit(&empty[s]);
                return true;
            };
            // ---------------------------------------------------------- issuer
            alive = alive && issue_rpart(base);
            for (int c = 0; c < nch && alive; ++c) {
                // chunk c's state-dependent steps, then the state-independent
                // steps of chunk c + 1 (queued behind them, they run while the
                // state threads update the state)
                if (!issue_dpart(base + c)) { alive = false; break; }
                if (c + 1 < nch && !issue_rpart(base + c + 1)) { alive = false; break; }
            }
        } else {
            // ---------------------------------------------------------- state
            float S[32];
            const float *src_state = first_seg ? init_block() : carry + sbase;
#pragma unroll
            for (int j = 0; j < 32; ++j)
                S[j] = src_state ? src_state[(size_t)(32 * qd + j) * kD + e] : 0.f;
            const uint32_t s_taddr = tm + lane_base + T2_S + 16 * qd;   // this thread's part of S^T
            write_state_tmem(s_taddr, S);
            fence_before_sync();
            mbar_arrive(&sready);
            for (int c = 0; c < nch && alive; ++c) {
                const int cc = base + c;
                // kGate: this chunk's gate values for the thread's output rows
                // [16 qd, 16 qd + 16) of column e, loaded before the waits so that
                // they arrive with the product; the gate then applies to the fp32
                // output before its one rounding to bf16
                uint32_t zg[kGate ? 16 : 1];
                if constexpr (kGate) {
                    const int tz = seq_t0 + (c_lo + c) * kC, Lz = min(kC, seq_t1 - tz);
                    const unsigned short *zrow = reinterpret_cast<const unsigned short *>(gate) +
                                                 ((size_t)(tz + 16 * qd) * H + h) * kD + e;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        zg[i] = 16 * qd + i < Lz && dbg_in(tz + 16 * qd + i, bd.tokens, kDbgTokenRow)
                                    ? zrow[(size_t)i * H * kD] : 0u;
                }
                // gamma has landed (its slot's barrier cannot run ahead: slot cc % 4
                // is refilled only after the product of chunk cc + 2, which needs
                // this thread's S^T of chunk cc + 1) and the chunk's product is in TMEM
                if (!wait_or_abort(&gfull[cc % kGamSlots], (cc / kGamSlots) & 1, abort_v, wait_limit) ||
                    !wait_or_abort(&sdone, cc & 1, abort_v, wait_limit)) {
                    alive = false;
                    break;
                }
                fence_after_sync();
                // S = gamma * S + P over this thread's 32 rows d, handed on as the next
                // S^T before this chunk's output is read (the next product waits
                // only for the state)
                {
                    const float *gam = reinterpret_cast<const float *>(sm + K2_GAM + (cc % kGamSlots) * 512) + 32 * qd;
#pragma unroll
                    for (int h16 = 0; h16 < 32; h16 += 16) {
                        float p[16];
                        tmem_ld16(tm + lane_base + T2_P + 256 * (cc & 1) + 32 * qd + h16, p);
                        tmem_ld_wait();
#pragma unroll
                        for (int j4 = 0; j4 < 16; j4 += 4) {
                            const int j = h16 + j4;
                            const float4 g4 = *reinterpret_cast<const float4 *>(gam + j);
                            const float2 s01 = __ffma2_rn(make_float2(g4.x, g4.y), make_float2(S[j], S[j + 1]),
                                                          make_float2(p[j4], p[j4 + 1]));
                            const float2 s23 = __ffma2_rn(make_float2(g4.z, g4.w), make_float2(S[j + 2], S[j + 3]),
                                                          make_float2(p[j4 + 2], p[j4 + 3]));
                            S[j] = s01.x; S[j + 1] = s01.y; S[j + 2] = s23.x; S[j + 3] = s23.y;
                        }
                        // this half of the next chunk's S^T, stored while the other half
                        // of P loads (workload 2 0.75% shorter than storing all of it
                        // after the update)
                        if (c + 1 < nch) {
                            float pk[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                pk[i] = __uint_as_float(pack_f16x2(S[h16 + 2 * i], S[h16 + 2 * i + 1]));
                            tmem_st8(s_taddr + h16 / 2, pk);
                        }
                    }
                }
                if (c + 1 < nch) {   // the next chunk's S^T complete (none after the chain's last chunk)
                    tmem_st_wait();
                    fence_before_sync();
                    mbar_arrive(&sready);
                }
                // output rows [16 qd, 16 qd + 16) of column e, rounded to bf16
                uint32_t ob16[8];
                {
                    float o[16];
                    tmem_ld16(tm + lane_base + T2_O + 256 * (cc & 1) + 16 * qd, o);
                    tmem_ld_wait();
                    fence_before_sync();
                    mbar_arrive(&pread[cc & 1]);   // P and O of the buffer read
                    if constexpr (kGate) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] = __fdividef(o[i], 1.f + __expf(-__uint_as_float(zg[i] << 16)));
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const __nv_bfloat162 v2 = __floats2bfloat162_rn(o[2 * j], o[2 * j + 1]);
                        ob16[j] = *reinterpret_cast<const uint32_t *>(&v2);
                    }
                }

                // this chunk's output, while the next state product runs: the warp's
                // 16 rows x 32 columns go through its own shared-memory tile (16-bit
                // stores, 64 contiguous bytes per row), and leave as 16-byte pieces
                // of rows, two stores per thread instead of sixteen 2-byte ones (the
                // narrow stores held the state warps' memory pipe: about 7% of a
                // one-chain call)
                const int t0 = seq_t0 + (c_lo + c) * kC;
                const int L = min(kC, seq_t1 - t0);
                {
                    unsigned short *ost = reinterpret_cast<unsigned short *>(sm + K2_OST + warp * 1024);
#pragma unroll
                    for (int rl2 = 0; rl2 < 8; ++rl2) {
                        ost[(2 * rl2) * 32 + lane] = (unsigned short)(ob16[rl2] & 0xFFFFu);
                        ost[(2 * rl2 + 1) * 32 + lane] = (unsigned short)(ob16[rl2] >> 16);
                    }
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int piece = lane + 32 * i, rl = piece >> 2, c8 = 8 * (piece & 3);   // row, 8 columns
                        const uint4 val = *reinterpret_cast<const uint4 *>(ost + rl * 32 + c8);
                        if (16 * qd + rl < L && dbg_in(t0 + 16 * qd + rl, bd.tokens, kDbgTokenRow))
                            *reinterpret_cast<uint4 *>(reinterpret_cast<unsigned short *>(out) +
                                                       ((size_t)(t0 + 16 * qd + rl) * H + h) * kD + 32 * q4 + c8) = val;
                    }
                    __syncwarp();   // the tile is rewritten for the next chunk
                }
                // checkpoint after every `stride` tokens of the sequence
                const int done = (c_lo + c) * kC + L;
                if (stride > 0 && io.ckpts && L == kC && done % stride == 0) {
                    const int64_t jc = (int64_t)tab.ckpt_off[n] + done / stride - 1;
                    const int64_t ps = jc < io.capacity ? pool_slot(io.ckpt_slots, jc, io.pool) : -1;
                    if (ps >= 0 && dbg_in(ps, bd.ckpts, kDbgCkpt)) {
                        float *dst = io.ckpts + ((size_t)ps * H + h) * DD + e;
#pragma unroll
                        for (int j = 0; j < 32; ++j) dst[(size_t)(32 * qd + j) * kD] = S[j];
                    }
                }
            }
            if (alive)
                if (float *dst_state = last_seg ? final_block() : carry + sbase) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) dst_state[(size_t)(32 * qd + j) * kD + e] = S[j];
                }
        }
        base_run += nch;
        if (!kMulti) break;
    }
    if (!alive) {
        *abort_v = 1;
        if (lane == 0) record_timeout(st);
    }
    // Never leave a copy or an MMA in flight (another role may have given up
    // while these two finished): the last stages' copies land, and a commit
    // arrives once every MMA the issuer started is complete.  After a normal
    // run both have already happened and the waits return at once.
    if (copier) {
        for (int c = max(0, copied_r - K2_STAGES); c < copied_r; ++c)
            mbar_wait_bounded(&fullr[c % K2_STAGES], (c / K2_STAGES) & 1, kDrainLimit);
        for (int c = max(0, copied - K2_STAGES); c < copied; ++c)
            mbar_wait_bounded(&full[c % K2_STAGES], (c / K2_STAGES) & 1, kDrainLimit);
        for (int c = max(0, copied_r - kGamSlots); c < copied_r; ++c)
            mbar_wait_bounded(&gfull[c % kGamSlots], (c / kGamSlots) & 1, kDrainLimit);
    }
    if (issuer) {
        mma_commit(&dbar);
        mbar_wait_bounded(&dbar, 0, kDrainLimit);
    }

    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tm, 512);
}

}  // namespace

size_t tc_handoff_bytes_per_chunk() { return REC_BYTES; }

// Streaming multiprocessors of the current device (read once per device); 152,
// a GB300's count, when no device can be queried (a host-only call without a
// GPU).
int64_t device_sm_count()
{
    constexpr int kDevs = 64;
    static std::atomic<int> cached[kDevs];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) {
        (void)cudaGetLastError();
        return 152;
    }
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            (void)cudaGetLastError();
            return 152;
        }
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

SegPlan tc_segment_plan(const kda_prefill_desc *d)
{
    // Many chains (sequences x heads): the recurrence alone would fill the GPU,
    // so it runs on a small persistent grid (kK2Share of the SMs, each CTA
    // taking chains one after another) while the preparation of the next
    // segment takes the other SMs.  Segments are uniform, kManyG chunks per
    // sequence (more where needed to stay within 64 segments), which bounds the
    // workspace to two ring slots of that many chunks of every chain.
    constexpr int64_t kManyG = 32, kManySegments = 64;
    constexpr double kK2Share = 0.26;
    // Automatic choice: overlap only when the recurrence (one CTA per chain and
    // SM) leaves most of the 152 SMs idle.  Segment lengths are whole K1 waves
    // (two K1 CTAs per SM; a wave covers 2 x SMs / chains chunks of every
    // sequence): the first segment, which K1 runs on all SMs before any K2,
    // four waves; then, on the SMs K2 leaves, segments of 16 waves, shrinking
    // towards the end (16, 13, 9, 6, 4, 2 waves) so that each K2 is shorter
    // than the K1 running beside it and the last K2, which nothing overlaps,
    // covers two waves only.  The segment just after the first takes the
    // remainder.  At most kMaxSegments segments (else uniform, as for an
    // explicit segment_chunks, which is raised to that bound where needed).
    constexpr int64_t kMaxChains = 96, kMinG = 4;
    const int64_t kSMs = device_sm_count();
    const int64_t T = d->total_tokens;
    const int64_t len = d->max_seq_len > 0 && d->max_seq_len < T ? d->max_seq_len : T;
    const int64_t maxc = (len + d->chunk - 1) / d->chunk;
    const int64_t chains = (int64_t)d->num_seqs * d->num_heads;
    SegPlan p{0, 1, 1, 0, {}};
    const int64_t k2_many = std::max<int64_t>(1, std::llround(kK2Share * (double)kSMs));
    auto finish = [&]() {
        p.G = 0;
        for (int s = 0; s < p.nseg; ++s) p.G = std::max(p.G, p.count(s));
        p.R = std::min(2, p.nseg);
        p.k2_ctas = 0;
        if (p.nseg > 1 && d->recurrence_ctas > 0) p.k2_ctas = (int)std::min<int64_t>(chains, d->recurrence_ctas);
        else if (p.nseg > 1 && chains > kMaxChains) p.k2_ctas = (int)std::min(chains, k2_many);
        return p;
    };
    if (d->segment_chunks == 0 && chains > kMaxChains) {
        const int64_t G = std::max(kManyG, (maxc + kManySegments - 1) / kManySegments);
        if (G >= maxc) return p;
        p.nseg = (int)((maxc + G - 1) / G);
        for (int s = 0; s <= p.nseg; ++s) p.lo[s] = (int)(s * G);
        return finish();
    }
    if (d->segment_chunks == 0) {
        if (chains <= 0) return p;
        const double wave_all = 2.0 * kSMs / chains, wave = 2.0 * (kSMs - chains) / chains;
        const int64_t first = std::max<int64_t>(kMinG, std::llround(4 * wave_all));
        if (first >= maxc) return p;
        static const int kTailWaves[] = {2, 4, 6, 9, 13, 16};
        int64_t tail[kMaxSegments], sum = 0;
        int nt = 0;
        while (first + sum < maxc && nt < kMaxSegments - 1) {
            const int w = nt < 6 ? kTailWaves[nt] : 16;
            tail[nt] = std::max<int64_t>(kMinG, std::llround(w * wave));
            sum += tail[nt++];
        }
        if (first + sum >= maxc) {
            // the earliest tail segment gives back the overshoot; one shorter than
            // kMinG joins the first segment instead
            int64_t head = first;
            tail[nt - 1] -= first + sum - maxc;
            if (tail[nt - 1] < kMinG) head += tail[--nt];
            p.nseg = 1 + nt;
            p.lo[0] = 0;
            p.lo[1] = (int)head;
            for (int s = 1; s < p.nseg; ++s) p.lo[s + 1] = p.lo[s] + (int)tail[nt - s];
            return finish();
        }
    }
    // uniform segments of G chunks (the last may reach past the sequence)
    int64_t G = d->segment_chunks > 0 ? d->segment_chunks : 1;
    G = std::max<int64_t>(G, (maxc + kMaxSegments - 1) / kMaxSegments);
    if (G >= maxc) return p;
    p.nseg = (int)((maxc + G - 1) / G);
    for (int s = 0; s <= p.nseg; ++s) p.lo[s] = (int)(s * G);
    return finish();
}

namespace {
thread_local char g_detail[256];

// Records the attributes of a kernel whose launch failed (for the error message).
template <typename F>
void note_launch_failure(F *fn, const char *name, int threads, uint32_t dyn_smem)
{
    cudaFuncAttributes at{};
    cudaFuncGetAttributes(&at, fn);
    snprintf(g_detail, sizeof g_detail,
             "%s: %d threads x %d registers (max %d threads per block), %zu B static + %u B dynamic smem",
             name, threads, at.numRegs, at.maxThreadsPerBlock, at.sharedSizeBytes, dyn_smem);
}

// The calling thread's side stream (highest priority: it carries the
// recurrence, the critical chain) and events on one device.  Created on first
// use and kept for the thread's lifetime.
constexpr int kRingMax = 2;
struct SideCtx {
    int device = -1;
    cudaStream_t side = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr, k1[kRingMax] = {}, k2[kRingMax] = {};
};
constexpr int kMaxDevices = 64;
thread_local SideCtx g_side[kMaxDevices];

cudaError_t side_ctx(SideCtx **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    SideCtx &c = g_side[dev];
    if (c.device != dev) {
        int lo = 0, hi = 0;
        if ((e = cudaDeviceGetStreamPriorityRange(&lo, &hi)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithPriority(&c.side, cudaStreamNonBlocking, hi)) != cudaSuccess) return e;
        const unsigned fl = cudaEventDisableTiming;
        if ((e = cudaEventCreateWithFlags(&c.fork, fl)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&c.join, fl)) != cudaSuccess) return e;
        for (int r = 0; r < kRingMax; ++r) {
            if ((e = cudaEventCreateWithFlags(&c.k1[r], fl)) != cudaSuccess) return e;
            if ((e = cudaEventCreateWithFlags(&c.k2[r], fl)) != cudaSuccess) return e;
        }
        c.device = dev;
    }
    *out = &c;
    return cudaSuccess;
}
// The kernels' shared-memory opt-in, once per device rather than on every call.
cudaError_t tc_kernel_attributes()
{
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t)1 << dev : 0;
    if (!bit || !(attr_done.load(std::memory_order_acquire) & bit)) {
        const void *k1s[] = {(const void *)k1_tc_kernel<false, 0>, (const void *)k1_tc_kernel<false, kH32>};
        for (const void *f : k1s)
            if ((e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)K1_SMEM)) != cudaSuccess)
                return e;
        const void *k1c[] = {(const void *)k1_tc_kernel<true, 0>, (const void *)k1_tc_kernel<true, kH32>};
        for (const void *f : k1c)
            if ((e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)(K1_SMEM + K1_TAPS_BYTES))) != cudaSuccess)
                return e;
        const void *k2s[] = {(const void *)k2_tc_kernel<false, false>, (const void *)k2_tc_kernel<true, false>,
                             (const void *)k2_tc_kernel<false, true>, (const void *)k2_tc_kernel<true, true>};
        for (const void *f : k2s)
            if ((e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)K2_SMEM)) != cudaSuccess)
                return e;
        attr_done.fetch_or(bit, std::memory_order_release);
    }
    return cudaSuccess;
}

// Per thread and device: a private stream on which a call's launches are
// captured, and a few executable graphs, one per launch structure (the number
// of segments, and whether K1 runs at all), reused least recently first.
constexpr int kGraphCache = 8;
struct GraphCtx {
    int device = -1;
    cudaStream_t cap = nullptr;
    int key[kGraphCache] = {};
    cudaGraphExec_t exec[kGraphCache] = {};
    uint64_t used[kGraphCache] = {}, tick = 0;
};
thread_local GraphCtx g_graph[kMaxDevices];
}  // namespace

const char *launch_failure_detail() { return g_detail; }

cudaError_t enqueue_prefill_tc(PrefillArgs a, cudaStream_t stream)
{
    a.stream = stream;
    cudaError_t e = cudaMemsetAsync(a.status, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
    if ((e = launch_seq_table(a)) != cudaSuccess) return e;
    if ((e = launch_prefill_tc(a)) != cudaSuccess) return e;
    return a.conv_out ? launch_conv_tail(a) : cudaSuccess;
}

cudaError_t launch_prefill_tc_graph(const PrefillArgs &a)
{
    // Everything a graph capture must not create is made first (the side
    // stream, its events, the kernels' attributes); then the call is captured
    // on this thread's private stream, the cached executable graph takes the
    // new launch parameters (or is instantiated again when the launch
    // structure changed) and is launched on the caller's stream.  When that
    // stream is itself being captured, or a graph call fails, the launches go
    // to the caller's stream directly.
    cudaError_t e;
    if ((e = tc_kernel_attributes()) != cudaSuccess) return e;
    SideCtx *c = nullptr;
    if ((e = side_ctx(&c)) != cudaSuccess) return e;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(a.stream, &cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return enqueue_prefill_tc(a, a.stream);
    }
    if (cs != cudaStreamCaptureStatusNone) return enqueue_prefill_tc(a, a.stream);
    GraphCtx &g = g_graph[c->device];
    if (g.device != c->device) {
        if (cudaStreamCreateWithFlags(&g.cap, cudaStreamNonBlocking) != cudaSuccess) {
            (void)cudaGetLastError();
            return enqueue_prefill_tc(a, a.stream);
        }
        g.device = c->device;
    }
    if (cudaStreamBeginCapture(g.cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        (void)cudaGetLastError();
        return enqueue_prefill_tc(a, a.stream);
    }
    e = enqueue_prefill_tc(a, g.cap);
    cudaGraph_t graph = nullptr;
    const cudaError_t ec = cudaStreamEndCapture(g.cap, &graph);
    if (e != cudaSuccess || ec != cudaSuccess || graph == nullptr) {
        if (graph) cudaGraphDestroy(graph);
        (void)cudaGetLastError();
        return e != cudaSuccess ? e : enqueue_prefill_tc(a, a.stream);
    }
    // the cached graph of this launch structure takes the new parameters; a
    // structure not cached replaces the least recently used graph
    const int key = 2 * a.plan.nseg + (a.max_chunks > 0 ? 1 : 0);
    int slot = -1, lru = 0;
    for (int i = 0; i < kGraphCache; ++i) {
        if (g.exec[i] && g.key[i] == key) slot = i;
        if (g.used[i] < g.used[lru]) lru = i;
    }
    cudaError_t r = cudaErrorInvalidValue;
    if (slot >= 0) {
        cudaGraphExecUpdateResultInfo info;
        r = cudaGraphExecUpdate(g.exec[slot], graph, &info);
        if (r != cudaSuccess) (void)cudaGetLastError();
    } else {
        slot = lru;
    }
    if (r != cudaSuccess) {
        if (g.exec[slot]) cudaGraphExecDestroy(g.exec[slot]);
        g.exec[slot] = nullptr;
        r = cudaGraphInstantiate(&g.exec[slot], graph, 0);
        if (r != cudaSuccess) g.exec[slot] = nullptr;
        g.key[slot] = key;
    }
    cudaGraphDestroy(graph);
    if (r != cudaSuccess) {
        (void)cudaGetLastError();
        return enqueue_prefill_tc(a, a.stream);
    }
    g.used[slot] = ++g.tick;
    return cudaGraphLaunch(g.exec[slot], a.stream);
}

namespace {
// One K1 launch (the plain or the convolving kernel).
void launch_k1(const PrefillArgs &a, unsigned grid, cudaStream_t stream, uint8_t *ring, int lo, int cnt, int G,
               int slot)
{
    const bf16 *q = (const bf16 *)a.q, *k = (const bf16 *)a.k, *v = (const bf16 *)a.v;
    const bool h32 = a.H == kH32;   // the common head count: strides fold into constants
    if (a.conv_w)
        (h32 ? k1_tc_kernel<true, kH32> : k1_tc_kernel<true, 0>)<<<grid, K1_THREADS, K1_SMEM + K1_TAPS_BYTES, stream>>>(
            q, k, v, a.g, a.beta, a.N, a.H, a.tab, ring, lo, cnt, G, slot, a.scalar_gate ? 1 : 0, a.status,
            a.wait_limit, a.conv_w, a.conv_width, a.conv_silu, (const bf16 *)a.conv_in, 0, a.bounds);
    else
        (h32 ? k1_tc_kernel<false, kH32> : k1_tc_kernel<false, 0>)<<<grid, K1_THREADS, K1_SMEM, stream>>>(
            q, k, v, a.g, a.beta, a.N, a.H, a.tab, ring, lo, cnt, G, slot, a.scalar_gate ? 1 : 0, a.status,
            a.wait_limit, nullptr, 0, 0, nullptr, (int)(device_sm_count() / 2), a.bounds);
}
// One K2 launch (one chain per CTA or chains in turn; with or without the gate).
void launch_k2(const PrefillArgs &a, bool multi, unsigned grid, cudaStream_t stream, const uint8_t *ring, int lo,
               int cnt, int G, int slot, float *carry)
{
    const bf16 *gate = (const bf16 *)a.gate;
    bf16 *out = (bf16 *)a.out;
    const StateIO io = state_io(a);
    if (multi && gate)
        k2_tc_kernel<true, true><<<grid, K2_THREADS, K2_SMEM, stream>>>(io, a.N, a.H, a.tab, ring, lo, cnt, G, slot,
                                                                         carry, out, a.status, a.wait_limit, gate, a.bounds);
    else if (multi)
        k2_tc_kernel<true, false><<<grid, K2_THREADS, K2_SMEM, stream>>>(io, a.N, a.H, a.tab, ring, lo, cnt, G, slot,
                                                                          carry, out, a.status, a.wait_limit, nullptr, a.bounds);
    else if (gate)
        k2_tc_kernel<false, true><<<grid, K2_THREADS, K2_SMEM, stream>>>(io, a.N, a.H, a.tab, ring, lo, cnt, G, slot,
                                                                          carry, out, a.status, a.wait_limit, gate, a.bounds);
    else
        k2_tc_kernel<false, false><<<grid, K2_THREADS, K2_SMEM, stream>>>(io, a.N, a.H, a.tab, ring, lo, cnt, G, slot,
                                                                           carry, out, a.status, a.wait_limit, nullptr, a.bounds);
}
}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs &a)
{
    cudaError_t e;
    g_detail[0] = 0;
    if ((e = tc_kernel_attributes()) != cudaSuccess) return e;
    uint8_t *ring = (uint8_t *)a.handoff;
    const unsigned chains = (unsigned)((size_t)a.N * a.H);
    const SegPlan &p = a.plan;

    if (p.nseg <= 1) {   // one K1 over every chunk, then one K2 over every sequence
        if (a.max_chunks > 0) {
            launch_k1(a, (unsigned)((size_t)a.max_chunks * a.H), a.stream, ring, 0, 0, 0, 0);
            if ((e = cudaGetLastError()) != cudaSuccess) {
                note_launch_failure(k1_tc_kernel<false, 0>, "K1", K1_THREADS, K1_SMEM);
                return e;
            }
        }
        launch_k2(a, false, chains, a.stream, ring, 0, 0, 0, 0, nullptr);
        if ((e = cudaGetLastError()) != cudaSuccess)
            note_launch_failure(k2_tc_kernel<false, false>, "K2", K2_THREADS, K2_SMEM);
        return e;
    }

    // Segments: K1(s) on the caller's stream, K2(s) on the side stream after
    // K1(s); K1(s) reuses ring slot s % R only after K2(s - R) has finished.
    SideCtx *c = nullptr;
    if ((e = side_ctx(&c)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(c->fork, a.stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(c->side, c->fork, 0)) != cudaSuccess) return e;
    for (int s = 0; s < p.nseg && e == cudaSuccess; ++s) {
        const int slot = s % p.R, lo = p.begin(s), cnt = p.count(s);
        const unsigned k1_grid = (unsigned)((size_t)a.N * cnt * a.H);
        if (s >= p.R && (e = cudaStreamWaitEvent(a.stream, c->k2[slot], 0)) != cudaSuccess) break;
        launch_k1(a, k1_grid, a.stream, ring, lo, cnt, p.G, slot);
        if ((e = cudaGetLastError()) != cudaSuccess) {
            note_launch_failure(k1_tc_kernel<false, 0>, "K1", K1_THREADS, K1_SMEM);
            break;
        }
        if ((e = cudaEventRecord(c->k1[slot], a.stream)) != cudaSuccess) break;
        if ((e = cudaStreamWaitEvent(c->side, c->k1[slot], 0)) != cudaSuccess) break;
        launch_k2(a, p.k2_ctas > 0, p.k2_ctas > 0 ? (unsigned)p.k2_ctas : chains, c->side, ring, lo, cnt, p.G, slot,
                  a.carry);
        if ((e = cudaGetLastError()) != cudaSuccess) {
            note_launch_failure(k2_tc_kernel<false, false>, "K2", K2_THREADS, K2_SMEM);
            break;
        }
        e = cudaEventRecord(c->k2[slot], c->side);
    }
    // join the side stream back, also after a failure (a stream capture needs it)
    cudaError_t ej = cudaEventRecord(c->join, c->side);
    if (ej == cudaSuccess) ej = cudaStreamWaitEvent(a.stream, c->join, 0);
    return e != cudaSuccess ? e : ej;
}

KDA_DBG_TAKE(dbg_take_prefill_tc)

}  // namespace kda
