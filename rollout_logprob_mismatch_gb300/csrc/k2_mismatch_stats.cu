// k2_mismatch_stats.cu -- segmented train/rollout mismatch statistics for sm_103a.
//
// Per token (VeXact summary eq. (1) and "KL Estimators"; llm-infra-atlas
// "训推一致性与 determinism" section 2; icarus "RL: Training Inference Mismatch",
// KL-estimator table and compute_consistency_and_kl_metrics; LoongSage
// "Train-Inference Consistency" sections 4-5):
//   delta = l_train - l_rollout, r = e^delta, k1 = -delta, k2 = delta^2 / 2,
//   k3 = (r - 1) - delta, w = min(r, C), clip = r > C, rel = |delta| / (|l_train| + 1e-8).
// Per sequence: means over its used tokens and the rejection flag (VeXact
// "Algorithmic TIM Compensation"); per batch: token means, mean of sequence means
// (icarus monitoring steps 2-3) and ratios.
//
// Two launches, in fp32 and integer arithmetic only (GB300 has very little
// fp64 throughput):
//  1. k2_seq_kernel, three 256-thread CTAs per SM.  A sequence of at most 8192
//     tokens is reduced by one warp (warps claim sequences in index order from
//     a counter), a longer one by a whole CTA.  Each warp
//     stages its sequence through shared memory in chunks of 448 tokens with 1-D
//     bulk copies (double-buffered: the next chunk is in flight while this one is
//     reduced), so a few instructions keep ~75 KB per SM in flight.  Inside a
//     chunk, lane i owns the tokens at index 64 p + i and 64 p + 32 + i
//     (p = 0..6), processed two at a time with packed f32x2 arithmetic and
//     summed in that order; chunks follow in order and each chunk's sums are
//     added to the lane's totals.  A fixed shuffle tree (and for a CTA a
//     warp-ordered sum) gives the sequence totals; the lanes of one warp write
//     the record.  The order depends only on a token's index inside its own
//     sequence and on the sequence's length, so a sequence's record has the same
//     bits wherever it is packed and whatever else is in the batch.
//  2. k2_fold_kernel: CTA j folds sequences 1024 j .. 1024 j + 1023 (4 per
//     thread, 16-word records) with float-float (TwoSum) sums and integer
//     counts in a fixed tree; the CTA that finishes last folds the partials.
// The batch record depends on S and the sequence records only.
#include <algorithm>
#include <cfloat>

#include "k2_internal.h"
#include "tim_internal.h"
#include "tim_ptx.cuh"
#include "../../include/tim.h"

namespace tim {
namespace {

enum { F_D = 0, F_AD, F_K2, F_K3, F_W, F_REL, NSUM };

// Sequence record, 16 words per sequence: word f of sequence s is rec[16 s + f].
enum {
    R_VALID = 0, R_N_MASK, R_N_USED, R_N_NAN, R_N_CLIP, R_FLAG,   // int32
    R_SD, R_SAD, R_SK2, R_SK3, R_SW, R_SREL, R_MAX, R_MK1, R_MK2, R_MK3,   // float
};
static_assert(R_MK3 + 1 == K2_REC_WORDS, "record layout");

// Fold partial: 7 int32 counts (N < 2^31), 9 float-float sums, 1 max (words).
enum { P_N_MASK = 0, P_N_USED, P_N_NAN, P_N_CLIP, P_NONEMPTY, P_REJ, P_INVALID, NCNT };
enum { S_SD = 0, S_SAD, S_SK2, S_SK3, S_SW, S_SREL, S_MK1, S_MK2, S_MK3, NDF };
static_assert(NCNT + 2 * NDF + 1 <= K2_PART_WORDS, "partial layout");

// Float-float value hi + lo and its addition (Knuth's TwoSum on the high
// parts, low parts added to the error term, renormalised).
struct ff {
    float hi, lo;
};

__device__ __forceinline__ ff ff_add(ff a, ff b)
{
    const float s = a.hi + b.hi;
    const float v = s - a.hi;
    float e = (a.hi - (s - v)) + (b.hi - v);
    e += a.lo + b.lo;
    const float hi = s + e;
    return {hi, e - (hi - s)};
}

__device__ __forceinline__ float qnan() { return __int_as_float(0x7fc00000); }

// Per-lane sums of one chunk (two tokens in lockstep: .x and .y) and the
// lane's running totals over chunks.
struct TokenAcc {
    float2 inner[NSUM];
    float outer[NSUM];
    float mx;
    int n_mask, n_used, n_clip;
};

__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }

// Two tokens at once (packed f32x2 arithmetic, round-to-nearest per component,
// so each component has the bits the scalar formula would give).  Tokens that
// are not used (masked out, past the chunk, or non-finite delta) contribute
// exact zeros.  Returns the two truncated IS weights (0 when not used).
__device__ __forceinline__ float2 token_pair(TokenAcc &t, float2 lt, float2 lr, bool m0, bool m1, float C,
                                             float lcd)
{
    const float2 d = __ffma2_rn(lr, f2(-1.f), lt);   // lt - lr, rounded once
    const bool f0 = fabsf(d.x) <= FLT_MAX, f1 = fabsf(d.y) <= FLT_MAX;   // false for inf, NaN
    const bool u0 = m0 && f0, u1 = m1 && f1;
    t.n_mask += static_cast<int>(m0) + static_cast<int>(m1);
    t.n_used += static_cast<int>(u0) + static_cast<int>(u1);   // n_nan = n_mask - n_used
    t.n_clip += static_cast<int>(u0 && d.x > lcd) + static_cast<int>(u1 && d.y > lcd);
    const float2 du = make_float2(u0 ? d.x : 0.f, u1 ? d.y : 0.f);
    const float2 ad = make_float2(fabsf(du.x), fabsf(du.y));
    const float2 e = __fmul2_rn(du, f2(1.4426950408889634f));   // e^d = 2^(d log2 e)
    const float2 r = make_float2(ex2(e.x), ex2(e.y));
    const float2 w = make_float2(u0 ? fminf(r.x, C) : 0.f, u1 ? fminf(r.y, C) : 0.f);
    const float2 dd = __fmul2_rn(du, du);
    // k3 = e^d - 1 - d: Taylor series sum_{n>=2} d^n / n! through n = 9 for
    // |d| < 0.5 (truncation below 2e-9 relative), (r - 1) - d above
    float2 p = f2(1.f / 362880.f);
    p = __ffma2_rn(p, du, f2(1.f / 40320.f));
    p = __ffma2_rn(p, du, f2(1.f / 5040.f));
    p = __ffma2_rn(p, du, f2(1.f / 720.f));
    p = __ffma2_rn(p, du, f2(1.f / 120.f));
    p = __ffma2_rn(p, du, f2(1.f / 24.f));
    p = __ffma2_rn(p, du, f2(1.f / 6.f));
    p = __ffma2_rn(p, du, f2(0.5f));
    const float2 small = __fmul2_rn(dd, p);
    const float2 large = __fadd2_rn(__fadd2_rn(r, f2(-1.f)), make_float2(-du.x, -du.y));
    const float2 k3 = make_float2(ad.x < 0.5f ? small.x : large.x, ad.y < 0.5f ? small.y : large.y);
    const float2 den = __fadd2_rn(make_float2(u0 ? fabsf(lt.x) : 1.f, u1 ? fabsf(lt.y) : 1.f), f2(1e-8f));
    const float2 rel = __fmul2_rn(ad, make_float2(rcp_approx(den.x), rcp_approx(den.y)));
    t.inner[F_D] = __fadd2_rn(t.inner[F_D], du);
    t.inner[F_AD] = __fadd2_rn(t.inner[F_AD], ad);
    t.inner[F_K2] = __ffma2_rn(dd, f2(0.5f), t.inner[F_K2]);
    t.inner[F_K3] = __fadd2_rn(t.inner[F_K3], k3);
    t.inner[F_W] = __fadd2_rn(t.inner[F_W], w);
    t.inner[F_REL] = __fadd2_rn(t.inner[F_REL], rel);
    t.mx = fmaxf(t.mx, fmaxf(ad.x, ad.y));
    return w;
}

// Totals of one sequence.
struct SeqTot {
    float sum[NSUM];
    int cnt[4];   // n_mask, n_used, n_nan, n_clip
    float mx;
};

// Where a staged chunk sits in its stage: tokens [t0, t0 + n) of the arrays,
// token t0 at float index off_f of the fp32 regions and byte off_m of the mask.
struct ChunkView {
    int64_t t0;   // first token of the chunk
    int n;        // tokens in the chunk
    int off_f;    // t0 & 3: index of token t0 in the staged fp32 regions
    int off_m;    // t0 & 15: byte of token t0 in the staged mask region
};

// Stages tokens [t0, t1) (at most K2_CHUNK) into the stage at `stp`: lane 0
// bulk-copies the 16-byte-aligned blocks that cover them (completion on
// `bar`); the few elements past the last whole 16-byte block of an array,
// which a bulk copy may not read, are copied by plain loads.  Called by a
// full warp.
__device__ __forceinline__ ChunkView stage_chunk(const K2Args &a, uint8_t *stp, uint32_t bar, int64_t t0,
                                                 int64_t t1, int lane, uint64_t pol)
{
    ChunkView v;
    v.t0 = t0;
    v.n = static_cast<int>(t1 - t0);
    v.off_f = static_cast<int>(t0 & 3);
    v.off_m = static_cast<int>(t0 & 15);
    const int64_t flim = a.N & ~int64_t(3);    // tokens below this lie in whole 16-byte fp32 blocks
    const int64_t mlim = a.N & ~int64_t(15);   // same for the mask bytes
    if (lane == 0) {
        const int64_t A = t0 & ~int64_t(3);
        const int64_t fend = min((t1 + 3) & ~int64_t(3), flim);
        const int fbytes = fend > A ? static_cast<int>(fend - A) * 4 : 0;
        const int64_t Am = t0 & ~int64_t(15);
        const int64_t mend = min((t1 + 15) & ~int64_t(15), mlim);
        const int mbytes = mend > Am ? static_cast<int>(mend - Am) : 0;
        const uint32_t st = smem_u32(stp);
        TIM_DCHECK(((reinterpret_cast<uintptr_t>(a.l_tr + A) | reinterpret_cast<uintptr_t>(a.mask + Am) |
                     static_cast<uintptr_t>(fbytes) | static_cast<uintptr_t>(mbytes)) & 15u) == 0u,
                   a.status, TIM_CHECK_BULK, t0, static_cast<uint64_t>(fbytes) << 32 | static_cast<uint32_t>(mbytes));
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, 2u * fbytes + mbytes);
        if (fbytes > 0) {
            bulk_load(st, a.l_tr + A, fbytes, bar, pol);
            bulk_load(st + K2_F_BYTES, a.l_ro + A, fbytes, bar, pol);
        }
        if (mbytes > 0)
            bulk_load(st + 2 * K2_F_BYTES, a.mask + Am, mbytes, bar, pol);
    }
    if (t1 > flim) {   // the last few elements of the arrays only
        float *lt_s = reinterpret_cast<float *>(stp) + v.off_f;
        float *lr_s = reinterpret_cast<float *>(stp + K2_F_BYTES) + v.off_f;
        for (int64_t t = max(t0, flim) + lane; t < t1; t += 32) {
            lt_s[t - t0] = a.l_tr[t];
            lr_s[t - t0] = a.l_ro[t];
        }
    }
    if (t1 > mlim) {
        uint8_t *mk_s = stp + 2 * K2_F_BYTES + v.off_m;
        for (int64_t t = max(t0, mlim) + lane; t < t1; t += 32)
            mk_s[t - t0] = a.mask[t];
    }
    return v;
}

// The lane's tokens of one staged chunk: index 64 q + lane (.x) and
// 64 q + 32 + lane (.y) for q = 0 .. K2_CHUNK / 64 - 1, in that order;
// writes their weights when WEIGHTS.
template <bool WEIGHTS>
__device__ __forceinline__ void reduce_chunk_t(TokenAcc &acc, const K2Args &a, const uint8_t *stp,
                                               const ChunkView &v, int lane)
{
    const float *lt_s = reinterpret_cast<const float *>(stp) + v.off_f + lane;
    const float *lr_s = reinterpret_cast<const float *>(stp + K2_F_BYTES) + v.off_f + lane;
    const uint8_t *mk_s = stp + 2 * K2_F_BYTES + v.off_m + lane;
    float *wout = WEIGHTS ? a.token_weight + v.t0 + lane : nullptr;
    TIM_DCHECK(v.t0 >= 0 && v.t0 + v.n <= a.N, a.status, TIM_CHECK_STORE, v.t0, v.n);
#ifdef TIM_DEBUG
    for (int j = lane; j < v.n; j += 32)   // mask bytes are 0 or 1
        TIM_DCHECK(mk_s[j - lane] <= 1, a.status, TIM_CHECK_MASK, v.t0 + j, mk_s[j - lane]);
#endif
    if (v.n == K2_CHUNK) {   // full chunk: no bounds checks
#pragma unroll
        for (int q = 0; q < K2_CHUNK / 64; ++q) {
            const float2 lt = make_float2(lt_s[64 * q], lt_s[64 * q + 32]);
            const float2 lr = make_float2(lr_s[64 * q], lr_s[64 * q + 32]);
            const float2 w = token_pair(acc, lt, lr, mk_s[64 * q] != 0, mk_s[64 * q + 32] != 0, a.C, a.log_c_down);
            if (WEIGHTS) {
                __stcs(wout + 64 * q, w.x);
                __stcs(wout + 64 * q + 32, w.y);
            }
        }
    } else {
#pragma unroll
        for (int q = 0; q < K2_CHUNK / 64; ++q) {
            const int j0 = 64 * q + lane, j1 = j0 + 32;
            const bool in0 = j0 < v.n, in1 = j1 < v.n;
            const float2 lt = make_float2(in0 ? lt_s[64 * q] : 0.f, in1 ? lt_s[64 * q + 32] : 0.f);
            const float2 lr = make_float2(in0 ? lr_s[64 * q] : 0.f, in1 ? lr_s[64 * q + 32] : 0.f);
            const bool m0 = in0 && mk_s[64 * q] != 0;
            const bool m1 = in1 && mk_s[64 * q + 32] != 0;
            const float2 w = token_pair(acc, lt, lr, m0, m1, a.C, a.log_c_down);
            if (WEIGHTS) {
                if (in0)
                    __stcs(wout + 64 * q, w.x);
                if (in1)
                    __stcs(wout + 64 * q + 32, w.y);
            }
        }
    }
}

__device__ __forceinline__ void reduce_chunk(TokenAcc &acc, const K2Args &a, const uint8_t *stp,
                                             const ChunkView &v, int lane)
{
    if (a.token_weight)
        reduce_chunk_t<true>(acc, a, stp, v, lane);
    else
        reduce_chunk_t<false>(acc, a, stp, v, lane);
}

// Adds the chunk's sums (at most 8 tokens per lane and half) into the lane's
// totals: two plain fp32 levels keep the rounding error within (8 + chunks) ulps.
__device__ __forceinline__ void fold_chunk(TokenAcc &acc)
{
#pragma unroll
    for (int f = 0; f < NSUM; ++f) {
        acc.outer[f] += acc.inner[f].x + acc.inner[f].y;
        acc.inner[f] = make_float2(0.f, 0.f);
    }
}

__device__ __forceinline__ SeqTot lane_total(const TokenAcc &acc)
{
    SeqTot t;
#pragma unroll
    for (int f = 0; f < NSUM; ++f)
        t.sum[f] = acc.outer[f];
    t.cnt[0] = acc.n_mask;
    t.cnt[1] = acc.n_used;
    t.cnt[2] = acc.n_mask - acc.n_used;   // a masked-in token is either used or non-finite
    t.cnt[3] = acc.n_clip;
    t.mx = acc.mx;
    return t;
}

__device__ __forceinline__ void acc_zero(TokenAcc &acc)
{
#pragma unroll
    for (int f = 0; f < NSUM; ++f) {
        acc.inner[f] = make_float2(0.f, 0.f);
        acc.outer[f] = 0.f;
    }
    acc.mx = 0.f;
    acc.n_mask = acc.n_used = acc.n_clip = 0;
}

// Fixed xor-shuffle tree over a warp; the result is taken from lane 0 and
// broadcast, so every lane holds the same bits.
__device__ __forceinline__ SeqTot warp_total(SeqTot t)
{
#pragma unroll
    for (int f = 0; f < NSUM; ++f) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            t.sum[f] += __shfl_xor_sync(0xffffffffu, t.sum[f], o);
        t.sum[f] = __shfl_sync(0xffffffffu, t.sum[f], 0);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c)
        t.cnt[c] = __reduce_add_sync(0xffffffffu, t.cnt[c]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        t.mx = fmaxf(t.mx, __shfl_xor_sync(0xffffffffu, t.mx, o));
    return t;
}

__device__ __forceinline__ float pick(const float (&v)[16], int i)
{
    float r = v[0];
#pragma unroll
    for (int k = 1; k < 16; ++k)
        r = i == k ? v[k] : r;
    return r;
}

// Means, flag, output record and workspace record of sequence s, written by
// one full warp whose lanes all hold the same totals (lane i writes word i).
__device__ __forceinline__ void write_seq(const K2Args &a, int s, const SeqTot &t, int lane)
{
    const float nu = static_cast<float>(t.cnt[1]);
    const float inv = t.cnt[1] > 0 ? 1.f / nu : 0.f;
    auto mean = [&](float x) { return x * inv; };
    const float md = mean(t.sum[F_D]);
    const float mk2 = mean(t.sum[F_K2]);
    const float mk3 = mean(t.sum[F_K3]);
    const int flag = t.cnt[1] > 0 && (a.estimator == 3 ? mk3 : fabsf(md)) > a.tau;
    float o[16];
    o[TIM_SEQ_N_MASK] = static_cast<float>(t.cnt[0]);
    o[TIM_SEQ_N_USED] = nu;
    o[TIM_SEQ_N_NAN] = static_cast<float>(t.cnt[2]);
    o[TIM_SEQ_N_CLIP] = static_cast<float>(t.cnt[3]);
    o[TIM_SEQ_MEAN_DELTA] = md;
    o[TIM_SEQ_MEAN_ABS_DELTA] = mean(t.sum[F_AD]);
    o[TIM_SEQ_MAX_ABS_DELTA] = t.mx;
    o[TIM_SEQ_MEAN_K1] = -md;
    o[TIM_SEQ_MEAN_K2] = mk2;
    o[TIM_SEQ_MEAN_K3] = mk3;
    o[TIM_SEQ_MEAN_W] = mean(t.sum[F_W]);
    o[TIM_SEQ_MEAN_REL] = mean(t.sum[F_REL]);
    o[12] = o[13] = o[14] = o[15] = 0.f;
    float *srow = a.seq_stats + static_cast<size_t>(s) * TIM_SEQ_FIELDS;
    if (a.stats_vec) {   // 16-byte aligned rows: three float4 stores
        if (lane < 3) {
            const float4 v = lane == 0 ? make_float4(o[0], o[1], o[2], o[3])
                           : lane == 1 ? make_float4(o[4], o[5], o[6], o[7])
                                       : make_float4(o[8], o[9], o[10], o[11]);
            reinterpret_cast<float4 *>(srow)[lane] = v;
        }
    } else if (lane < TIM_SEQ_FIELDS) {
        srow[lane] = pick(o, lane);
    }
    uint32_t r[16];
    r[R_VALID] = 1u;
    r[R_N_MASK] = static_cast<uint32_t>(t.cnt[0]);
    r[R_N_USED] = static_cast<uint32_t>(t.cnt[1]);
    r[R_N_NAN] = static_cast<uint32_t>(t.cnt[2]);
    r[R_N_CLIP] = static_cast<uint32_t>(t.cnt[3]);
    r[R_FLAG] = static_cast<uint32_t>(flag);
    r[R_SD] = __float_as_uint(t.sum[F_D]);
    r[R_SAD] = __float_as_uint(t.sum[F_AD]);
    r[R_SK2] = __float_as_uint(t.sum[F_K2]);
    r[R_SK3] = __float_as_uint(t.sum[F_K3]);
    r[R_SW] = __float_as_uint(t.sum[F_W]);
    r[R_SREL] = __float_as_uint(t.sum[F_REL]);
    r[R_MAX] = __float_as_uint(t.mx);
    r[R_MK1] = __float_as_uint(-md);
    r[R_MK2] = __float_as_uint(mk2);
    r[R_MK3] = __float_as_uint(mk3);
    if (lane < 4) {
        const uint4 v = lane == 0 ? make_uint4(r[0], r[1], r[2], r[3])
                      : lane == 1 ? make_uint4(r[4], r[5], r[6], r[7])
                      : lane == 2 ? make_uint4(r[8], r[9], r[10], r[11])
                                  : make_uint4(r[12], r[13], r[14], r[15]);
        reinterpret_cast<uint4 *>(a.rec + static_cast<size_t>(s) * K2_REC_WORDS)[lane] = v;
    }
    if (lane == 0)
        a.seq_flags[s] = flag;
}

struct FoldAcc {
    int cnt[NCNT];
    ff sum[NDF];
    float mx;
};

__device__ __forceinline__ void fold_zero(FoldAcc &f)
{
#pragma unroll
    for (int i = 0; i < NCNT; ++i)
        f.cnt[i] = 0;
#pragma unroll
    for (int i = 0; i < NDF; ++i)
        f.sum[i] = {0.f, 0.f};
    f.mx = 0.f;
}

__device__ __forceinline__ void fold_add(FoldAcc &x, const FoldAcc &y)
{
#pragma unroll
    for (int i = 0; i < NCNT; ++i)
        x.cnt[i] += y.cnt[i];
#pragma unroll
    for (int i = 0; i < NDF; ++i)
        x.sum[i] = ff_add(x.sum[i], y.sum[i]);
    x.mx = fmaxf(x.mx, y.mx);
}

// One level of a fixed xor-shuffle tree: x += x of lane ^ o, field by field
// (the float-float sum is symmetric, so both lanes get the same bits).
__device__ __forceinline__ void fold_shfl_add(FoldAcc &x, int o)
{
#pragma unroll
    for (int i = 0; i < NCNT; ++i)
        x.cnt[i] += __shfl_xor_sync(0xffffffffu, x.cnt[i], o);
#pragma unroll
    for (int i = 0; i < NDF; ++i) {
        const ff y = {__shfl_xor_sync(0xffffffffu, x.sum[i].hi, o), __shfl_xor_sync(0xffffffffu, x.sum[i].lo, o)};
        x.sum[i] = ff_add(x.sum[i], y);
    }
    x.mx = fmaxf(x.mx, __shfl_xor_sync(0xffffffffu, x.mx, o));
}

// The warp's total, on lane 0 (and on every lane): a fixed tree.
__device__ __forceinline__ void fold_warp(FoldAcc &x)
{
#pragma unroll 1
    for (int o = 16; o > 0; o >>= 1)
        fold_shfl_add(x, o);
}

__device__ __forceinline__ void fold_store(uint32_t *p, const FoldAcc &f)
{
    for (int i = 0; i < NCNT; ++i)
        p[i] = static_cast<uint32_t>(f.cnt[i]);
    for (int i = 0; i < NDF; ++i) {
        p[NCNT + 2 * i] = __float_as_uint(f.sum[i].hi);
        p[NCNT + 2 * i + 1] = __float_as_uint(f.sum[i].lo);
    }
    p[NCNT + 2 * NDF] = __float_as_uint(f.mx);
}

// From shared memory.
__device__ __forceinline__ void fold_load(FoldAcc &f, const uint32_t *p)
{
#pragma unroll
    for (int i = 0; i < NCNT; ++i)
        f.cnt[i] = static_cast<int>(p[i]);
#pragma unroll
    for (int i = 0; i < NDF; ++i)
        f.sum[i] = {__uint_as_float(p[NCNT + 2 * i]), __uint_as_float(p[NCNT + 2 * i + 1])};
    f.mx = __uint_as_float(p[NCNT + 2 * NDF]);
}

// From global memory written by another CTA (read through L2).
__device__ __forceinline__ void fold_load_global(FoldAcc &f, const uint32_t *p)
{
#pragma unroll
    for (int i = 0; i < NCNT; ++i)
        f.cnt[i] = static_cast<int>(__ldcg(p + i));
#pragma unroll
    for (int i = 0; i < NDF; ++i)
        f.sum[i] = {__uint_as_float(__ldcg(p + NCNT + 2 * i)), __uint_as_float(__ldcg(p + NCNT + 2 * i + 1))};
    f.mx = __uint_as_float(__ldcg(p + NCNT + 2 * NDF));
}

// fp32 -> fp64 by moving bits (exact; fp32 subnormals are renormalised).  The
// batch record is written without fp64 arithmetic, which GB300 runs slowly.
__device__ __forceinline__ double widen(float f)
{
    const uint32_t u = __float_as_uint(f);
    const uint64_t sign = static_cast<uint64_t>(u >> 31) << 63;
    const uint32_t e = (u >> 23) & 0xffu, m = u & 0x7fffffu;
    uint64_t bits;
    if (e == 0u && m == 0u) {
        bits = sign;
    } else if (e == 0u) {
        const int msb = 31 - __clz(static_cast<int>(m));   // value = m * 2^-149
        bits = sign | (static_cast<uint64_t>(msb - 149 + 1023) << 52) |
               ((static_cast<uint64_t>(m) << (52 - msb)) & ((uint64_t(1) << 52) - 1));
    } else if (e == 255u) {
        bits = sign | (uint64_t(0x7ff) << 52) | (static_cast<uint64_t>(m) << 29);
    } else {
        bits = sign | (static_cast<uint64_t>(e - 127 + 1023) << 52) | (static_cast<uint64_t>(m) << 29);
    }
    return __longlong_as_double(static_cast<long long>(bits));
}

// A count (< 2^31) as fp64, by moving bits.
__device__ __forceinline__ double widen_count(long long n)
{
    if (n <= 0)
        return 0.0;
    const uint64_t v = static_cast<uint64_t>(n);
    const int lz = __clzll(static_cast<long long>(v));
    const uint64_t frac = ((v << lz) << 1) >> 12;
    return __longlong_as_double(static_cast<long long>((static_cast<uint64_t>(63 - lz + 1023) << 52) | frac));
}

// The batch record from the folded totals (thread 0).  Means and ratios are
// fp32 quotients (relative error ~1e-7) of the float-float sums and counts.
__device__ void write_batch(const K2Args &a, const FoldAcc &t, bool check_offsets)
{
    bool bad = t.cnt[P_INVALID] > 0;
    if (check_offsets)
        bad = bad || a.off[0] != 0 || static_cast<int64_t>(a.off[a.S]) != a.N;
    if (bad)
        atomicCAS(a.status, 0, static_cast<int>(TIM_ERR_BAD_INPUT));
    const float n_used = static_cast<float>(t.cnt[P_N_USED]);
    const float n_ne = static_cast<float>(t.cnt[P_NONEMPTY]);
    const float n_mask = static_cast<float>(t.cnt[P_N_MASK]);
    auto mean = [&](int i, float n) { return n > 0.f ? widen((t.sum[i].hi + t.sum[i].lo) / n) : 0.0; };
    auto ratio = [](int x, float n) { return n > 0.f ? widen(static_cast<float>(x) / n) : 0.0; };
    double *o = a.batch;
    o[TIM_BATCH_N_MASK] = widen_count(t.cnt[P_N_MASK]);
    o[TIM_BATCH_N_USED] = widen_count(t.cnt[P_N_USED]);
    o[TIM_BATCH_N_NAN] = widen_count(t.cnt[P_N_NAN]);
    o[TIM_BATCH_N_CLIP] = widen_count(t.cnt[P_N_CLIP]);
    o[TIM_BATCH_MEAN_DELTA] = mean(S_SD, n_used);
    o[TIM_BATCH_MEAN_ABS_DELTA] = mean(S_SAD, n_used);
    o[TIM_BATCH_MAX_ABS_DELTA] = widen(t.mx);
    o[TIM_BATCH_MEAN_K1] = n_used > 0.f ? widen(-((t.sum[S_SD].hi + t.sum[S_SD].lo) / n_used)) : 0.0;
    o[TIM_BATCH_MEAN_K2] = mean(S_SK2, n_used);
    o[TIM_BATCH_MEAN_K3] = mean(S_SK3, n_used);
    o[TIM_BATCH_MEAN_W] = mean(S_SW, n_used);
    o[TIM_BATCH_MEAN_REL] = mean(S_SREL, n_used);
    o[TIM_BATCH_SEQMEAN_K1] = mean(S_MK1, n_ne);
    o[TIM_BATCH_SEQMEAN_K2] = mean(S_MK2, n_ne);
    o[TIM_BATCH_SEQMEAN_K3] = mean(S_MK3, n_ne);
    o[TIM_BATCH_CLIP_RATIO] = ratio(t.cnt[P_N_CLIP], n_mask);
    o[TIM_BATCH_NAN_RATIO] = ratio(t.cnt[P_N_NAN], n_mask);
    o[TIM_BATCH_REJECT_RATIO] = ratio(t.cnt[P_REJ], n_ne);
    o[TIM_BATCH_N_SEQS_NONEMPTY] = widen_count(t.cnt[P_NONEMPTY]);
    o[TIM_BATCH_N_REJECTED] = widen_count(t.cnt[P_REJ]);
    if (bad)
        for (int f = 0; f < TIM_BATCH_FIELDS; ++f)
            o[f] = __longlong_as_double(0x7ff8000000000000ll);
}

// The fold term of sequence s (its 16-word record, read through L2: other
// warps wrote it).
// One sequence record (16 words, loaded as four 16-byte words) folded into x.
__device__ __forceinline__ void fold_rec(FoldAcc &x, const uint4 (&q)[4])
{
    const uint32_t rc[16] = {q[0].x, q[0].y, q[0].z, q[0].w, q[1].x, q[1].y, q[1].z, q[1].w,
                             q[2].x, q[2].y, q[2].z, q[2].w, q[3].x, q[3].y, q[3].z, q[3].w};
    FoldAcc y;
    fold_zero(y);
    if (rc[R_VALID] == 0u) {
        y.cnt[P_INVALID] = 1;
    } else {
        const uint32_t nu = rc[R_N_USED];
        y.cnt[P_N_MASK] = static_cast<int>(rc[R_N_MASK]);
        y.cnt[P_N_USED] = static_cast<int>(nu);
        y.cnt[P_N_NAN] = static_cast<int>(rc[R_N_NAN]);
        y.cnt[P_N_CLIP] = static_cast<int>(rc[R_N_CLIP]);
        y.sum[S_SD] = {__uint_as_float(rc[R_SD]), 0.f};
        y.sum[S_SAD] = {__uint_as_float(rc[R_SAD]), 0.f};
        y.sum[S_SK2] = {__uint_as_float(rc[R_SK2]), 0.f};
        y.sum[S_SK3] = {__uint_as_float(rc[R_SK3]), 0.f};
        y.sum[S_SW] = {__uint_as_float(rc[R_SW]), 0.f};
        y.sum[S_SREL] = {__uint_as_float(rc[R_SREL]), 0.f};
        y.mx = __uint_as_float(rc[R_MAX]);
        if (nu > 0u) {
            y.cnt[P_NONEMPTY] = 1;
            y.cnt[P_REJ] = static_cast<int>(rc[R_FLAG]);
            y.sum[S_MK1] = {__uint_as_float(rc[R_MK1]), 0.f};
            y.sum[S_MK2] = {__uint_as_float(rc[R_MK2]), 0.f};
            y.sum[S_MK3] = {__uint_as_float(rc[R_MK3]), 0.f};
        }
    }
    fold_add(x, y);
}

__device__ __forceinline__ bool offsets_ok(const K2Args &a, int s, int64_t b, int64_t e)
{
    bool ok = b >= 0 && e >= b && e <= a.N;
    if (s == 0 && b != 0)
        ok = false;
    if (s == a.S - 1 && e != a.N)
        ok = false;
    return ok;
}

// Bounded wait on a stage barrier; raises the CTA's abort flag on expiry.
__device__ __forceinline__ bool stage_wait(uint32_t bar, uint32_t parity, volatile int *abort, uint64_t budget)
{
    return mbar_wait_sleep(bar, parity, abort, budget);
}

// Lane-parallel record of a sequence that is skipped by the staged path:
// bad offsets (NaN record, status) or no tokens (all zero).
__device__ __forceinline__ void write_plain(const K2Args &a, int s, bool bad, int lane)
{
    if (bad) {
        if (lane == 0)
            atomicCAS(a.status, 0, static_cast<int>(TIM_ERR_BAD_INPUT));
        if (lane < TIM_SEQ_FIELDS)
            a.seq_stats[static_cast<size_t>(s) * TIM_SEQ_FIELDS + lane] = qnan();
        if (lane < K2_REC_WORDS)
            a.rec[static_cast<size_t>(s) * K2_REC_WORDS + lane] = 0u;   // not valid
        if (lane == 0)
            a.seq_flags[s] = 0;
    } else {
        SeqTot z;
#pragma unroll
        for (int f = 0; f < NSUM; ++f)
            z.sum[f] = 0.f;
        z.cnt[0] = z.cnt[1] = z.cnt[2] = z.cnt[3] = 0;
        z.mx = 0.f;
        write_seq(a, s, z, lane);
    }
}

// Claims the warp's next ticket (lane 0 takes it from the call's counter;
// the value is not waited for until it is broadcast).
__device__ __forceinline__ int claim_raw(const K2Args &a, int lane)
{
    return lane == 0 ? atomicAdd(a.claim, 1) : 0;
}

// The sequences of ticket t: the first t0 = block_tickets(S) tickets hand out
// K2_CLAIM_BLOCK consecutive sequences each, the later ones one each.  The
// blocks cut the counter's traffic (one claim per sequence from every warp
// queued on the counter's word, and how long varied from one device to
// another); single sequences at the end keep the warps' finish times close,
// and a batch of few sequences (at most two per warp of the grid) goes out
// one sequence at a time, spread over as many warps as it can.
__device__ __forceinline__ int block_tickets(int S)
{
    const int singles = min(S, max(S / 8, 2 * static_cast<int>(gridDim.x) * K2_WARPS));
    return (S - singles) / K2_CLAIM_BLOCK;
}

__device__ __forceinline__ void ticket_range(int t, int S, int t0, int &lo, int &hi)
{
    if (t < t0) {
        lo = t * K2_CLAIM_BLOCK;
        hi = lo + K2_CLAIM_BLOCK;
    } else {
        lo = t0 * K2_CLAIM_BLOCK + (t - t0);   // t < S + (claims in flight): no overflow
        hi = lo + 1;
    }
    hi = min(hi, S);
}

// The next sequence the warp reduces itself, from the range [cur, end) of its
// current ticket; when that is used up, the ticket claimed one range earlier
// (lane 0: pend) gives the next range and a new ticket is claimed, so a
// claim's latency hides behind the sequences before it.  Records of empty or
// bad sequences met on the way are written at once, long ones are left for
// the CTA phase.  Returns S when there is none (every later ticket is past S
// too).
__device__ __forceinline__ int next_short(const K2Args &a, int t0, int &cur, int &end, int &pend, int lane)
{
    while (true) {
        if (cur >= end) {
            const int t = __shfl_sync(0xffffffffu, pend, 0);
            pend = claim_raw(a, lane);
            ticket_range(t, a.S, t0, cur, end);
            if (cur >= a.S)
                return a.S;
        }
        const int s = cur++;
        const int64_t b = a.off[s], e = a.off[s + 1];
        if (!offsets_ok(a, s, b, e)) {
            write_plain(a, s, true, lane);
            continue;
        }
        if (e - b > K2_LONG)
            continue;
        if (e == b) {
            write_plain(a, s, false, lane);
            continue;
        }
        return s;
    }
}

__global__ void __launch_bounds__(K2_THREADS, K2_CTAS_PER_SM) k2_seq_kernel(const K2Args a)
{
    extern __shared__ __align__(16) uint8_t k2_smem[];
    __shared__ float red_f[K2_WARPS][NSUM];
    __shared__ int red_i[K2_WARPS][4];
    __shared__ float red_mx[K2_WARPS];
    __shared__ int abort_flag_s;
    volatile int *abort_flag = &abort_flag_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t bar0 = smem_u32(k2_smem) + 8u * (K2_STAGES * warp);
    uint8_t *const st0 = k2_smem + K2_BAR_BYTES + K2_STAGES * K2_STAGE_BYTES * warp;
    if (lane == 0) {
        for (int i = 0; i < K2_STAGES; ++i)
            mbar_init(bar0 + 8u * i, 1);
        fence_mbar_init();
    }
    if (tid == 0)
        abort_flag_s = 0;
    pdl_wait();                // the inputs may be written by the previous kernel
    pdl_launch_dependents();   // the fold kernel may start launching
    // Does this CTA have a sequence longer than K2_LONG (phase 2)?  Most batches
    // have none, and then no warp waits for the others at the phase boundary.
    bool mine = false;
    for (int q = blockIdx.x + tid * gridDim.x; q < a.S; q += K2_THREADS * gridDim.x) {
        const int64_t b = a.off[q], e = a.off[q + 1];
        mine = mine || (offsets_ok(a, q, b, e) && e - b > K2_LONG);
    }
    const bool has_long = __syncthreads_or(mine) != 0;
    const uint64_t pol = l2_policy_evict_first();
    const uint64_t budget = a.wait_budget_ns;
    uint32_t parity = 0;    // bit i: parity of stage i's next completion
    uint32_t pending = 0;   // bit i: stage i has a staged chunk not yet waited for
    int stage = 0;
    bool ok = true;

    // ---- phase 1: sequences of at most K2_LONG tokens, one warp each.  Warps
    // claim sequences in index order from the call's counter, one ticket ahead
    // of the range they reduce, so the work stays balanced however the lengths
    // vary (a record's bits depend on its own tokens only, not on the warp
    // that reduces it).
    const int t0 = block_tickets(a.S);
    int pend = claim_raw(a, lane), t_cur = 0, t_end = 0;   // lane 0: the next ticket; the current range
    int s = next_short(a, t0, t_cur, t_end, pend, lane);
    ChunkView cur;
    if (s < a.S) {
        const int64_t b = a.off[s], e = a.off[s + 1];
        cur = stage_chunk(a, st0, bar0, b, min(e, b + K2_CHUNK), lane, pol);
        pending |= 1u;
    }
    while (ok && s < a.S) {
        const int64_t b = a.off[s], e = a.off[s + 1];
        const int64_t nch = (e - b + K2_CHUNK - 1) / K2_CHUNK;
        TokenAcc acc;
        acc_zero(acc);
        int nxt = s;
        for (int64_t c = 0; c < nch; ++c) {
            ChunkView nv;
            uint8_t *const nst = st0 + (stage ^ 1) * K2_STAGE_BYTES;
            const uint32_t nbar = bar0 + 8u * (stage ^ 1);
            if (c + 1 < nch) {
                const int64_t t0 = b + (c + 1) * K2_CHUNK;
                nv = stage_chunk(a, nst, nbar, t0, min(e, t0 + K2_CHUNK), lane, pol);
                pending |= 1u << (stage ^ 1);
            } else {
                nxt = next_short(a, t0, t_cur, t_end, pend, lane);
                if (nxt < a.S) {
                    const int64_t nb = a.off[nxt], ne = a.off[nxt + 1];
                    nv = stage_chunk(a, nst, nbar, nb, min(ne, nb + K2_CHUNK), lane, pol);
                    pending |= 1u << (stage ^ 1);
                }
            }
            if (!stage_wait(bar0 + 8u * stage, (parity >> stage) & 1u, abort_flag, budget)) {
                ok = false;
                break;
            }
            parity ^= 1u << stage;
            pending &= ~(1u << stage);
            reduce_chunk(acc, a, st0 + stage * K2_STAGE_BYTES, cur, lane);
            fold_chunk(acc);
            __syncwarp();
            stage ^= 1;
            cur = nv;
        }
        if (!ok)
            break;
        write_seq(a, s, warp_total(lane_total(acc)), lane);
        s = nxt;
    }
    if (!ok) {
        // staged copies may still be landing: give them their time before the CTA exits
        for (int i = 0; i < K2_STAGES; ++i)
            if (pending & (1u << i))
                drain_wait(bar0 + 8u * i, (parity >> i) & 1u);
        pending = 0;
        if (lane == 0)
            atomicCAS(a.status, 0, static_cast<int>(TIM_ERR_TIMEOUT));
    }

    // ---- phase 2: longer sequences, one CTA each; warp w takes chunks w, w + K2_WARPS, ...
    // (the sequences q = blockIdx.x + k gridDim.x; phase 1 skipped every long one)
    if (!has_long)   // uniform over the CTA
        return;
    if (!ok)
        *abort_flag = 1;
    __syncthreads();
    for (int q = blockIdx.x; q < a.S && !*abort_flag; q += gridDim.x) {
        const int64_t b = a.off[q], e = a.off[q + 1];
        if (!offsets_ok(a, q, b, e) || e - b <= K2_LONG)   // uniform over the CTA
            continue;
        __syncthreads();   // the previous long sequence's reduction buffers are free
        const int64_t nch = (e - b + K2_CHUNK - 1) / K2_CHUNK;
        TokenAcc acc;
        acc_zero(acc);
        int64_t c = warp;
        if (c < nch) {
            cur = stage_chunk(a, st0 + stage * K2_STAGE_BYTES, bar0 + 8u * stage,
                              b + c * K2_CHUNK, min(e, b + (c + 1) * K2_CHUNK), lane, pol);
            pending |= 1u << stage;
        }
        for (; c < nch; c += K2_WARPS) {
            ChunkView nv;
            const int64_t cn = c + K2_WARPS;
            if (cn < nch) {
                nv = stage_chunk(a, st0 + (stage ^ 1) * K2_STAGE_BYTES,
                                 bar0 + 8u * (stage ^ 1), b + cn * K2_CHUNK, min(e, b + (cn + 1) * K2_CHUNK),
                                 lane, pol);
                pending |= 1u << (stage ^ 1);
            }
            if (!stage_wait(bar0 + 8u * stage, (parity >> stage) & 1u, abort_flag, budget)) {
                ok = false;
                break;
            }
            parity ^= 1u << stage;
            pending &= ~(1u << stage);
            reduce_chunk(acc, a, st0 + stage * K2_STAGE_BYTES, cur, lane);
            fold_chunk(acc);
            __syncwarp();
            stage ^= 1;
            cur = nv;
        }
        if (!ok) {
            for (int i = 0; i < K2_STAGES; ++i)
                if (pending & (1u << i))
                    drain_wait(bar0 + 8u * i, (parity >> i) & 1u);
            pending = 0;
            if (lane == 0)
                atomicCAS(a.status, 0, static_cast<int>(TIM_ERR_TIMEOUT));
        }
        const SeqTot t = warp_total(lane_total(acc));
        if (lane == 0) {
#pragma unroll
            for (int f = 0; f < NSUM; ++f)
                red_f[warp][f] = t.sum[f];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                red_i[warp][k] = t.cnt[k];
            red_mx[warp] = t.mx;
        }
        __syncthreads();
        if (warp == 0) {   // every lane folds the warps in order: the same bits on all lanes
            SeqTot c2;
#pragma unroll
            for (int f = 0; f < NSUM; ++f)
                c2.sum[f] = 0.f;
            c2.cnt[0] = c2.cnt[1] = c2.cnt[2] = c2.cnt[3] = 0;
            c2.mx = 0.f;
            for (int w = 0; w < K2_WARPS; ++w) {
#pragma unroll
                for (int f = 0; f < NSUM; ++f)
                    c2.sum[f] += red_f[w][f];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    c2.cnt[k] += red_i[w][k];
                c2.mx = fmaxf(c2.mx, red_mx[w]);
            }
            write_seq(a, q, c2, lane);
        }
    }
}

// Fold of the sequence records into the batch record, one launch: CTA b folds
// sequences 1024 b .. 1024 b + 1023 -- thread i takes 1024 b + i + 256 k for
// k = 0..3 in order, a fixed xor tree per warp, then warp 0 adds the 8 warp
// totals in warp order -- into the block's partial; the CTA that finishes
// last (a ticket) folds the partials the same way (thread i: partials i,
// i + 256, ...).  The order of every sum is fixed by S alone.
__device__ __forceinline__ FoldAcc fold_cta(FoldAcc x)
{
    __shared__ uint32_t sh[K2_FOLD_THREADS / 32][K2_PART_WORDS];
    fold_warp(x);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0)
        fold_store(sh[warp], x);
    __syncthreads();
    FoldAcc t;
    fold_zero(t);
    if (warp == 0 && lane == 0)
        for (int w = 0; w < K2_FOLD_THREADS / 32; ++w) {
            FoldAcc y;
            fold_load(y, sh[w]);
            fold_add(t, y);
        }
    return t;   // on thread 0
}

__global__ void __launch_bounds__(K2_FOLD_THREADS) k2_fold_kernel(const K2Args a)
{
    pdl_wait();   // the records come from k2_seq_kernel
    __shared__ int last_s;
    FoldAcc x;
    fold_zero(x);
    // the thread's records s0, s0 + K2_FOLD_THREADS, ...: all loaded first,
    // then folded in that order
    constexpr int PER = K2_FOLD_SEQS / K2_FOLD_THREADS;
    const int64_t s1 = min(static_cast<int64_t>(a.S), static_cast<int64_t>(blockIdx.x + 1) * K2_FOLD_SEQS);
    const int64_t s0 = static_cast<int64_t>(blockIdx.x) * K2_FOLD_SEQS + threadIdx.x;
    uint4 q[PER][4];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int64_t s = s0 + static_cast<int64_t>(k) * K2_FOLD_THREADS;
        if (s < s1) {
            const uint4 *rp = reinterpret_cast<const uint4 *>(a.rec + static_cast<size_t>(s) * K2_REC_WORDS);
#pragma unroll
            for (int w = 0; w < 4; ++w)
                q[k][w] = __ldcg(rp + w);
        }
    }
#pragma unroll
    for (int k = 0; k < PER; ++k)
        if (s0 + static_cast<int64_t>(k) * K2_FOLD_THREADS < s1)
            fold_rec(x, q[k]);
    const FoldAcc t = fold_cta(x);
    if (threadIdx.x == 0) {
        if (gridDim.x == 1) {
            write_batch(a, t, false);
            last_s = 0;
        } else {
            fold_store(a.part + static_cast<size_t>(blockIdx.x) * K2_PART_WORDS, t);
            __threadfence();
            last_s = atomicAdd(a.blk_done, 1) == static_cast<int>(gridDim.x) - 1;
        }
    }
    __syncthreads();
    if (!last_s)
        return;
    __threadfence();   // every CTA's partial is visible
    FoldAcc y;
    fold_zero(y);
    for (int p = threadIdx.x; p < static_cast<int>(gridDim.x); p += K2_FOLD_THREADS) {
        FoldAcc z;
        fold_load_global(z, a.part + static_cast<size_t>(p) * K2_PART_WORDS);
        fold_add(y, z);
    }
    const FoldAcc f = fold_cta(y);
    if (threadIdx.x == 0)
        write_batch(a, f, false);
}

// S = 0: only the (all-zero) batch record, after checking the offsets cover
// [0, N) when there are offsets.
__global__ void k2_empty_kernel(const K2Args a)
{
    FoldAcc t;
    fold_zero(t);
    write_batch(a, t, a.off != nullptr);
}

} // namespace

cudaError_t k2_prepare_device()
{
    return cudaFuncSetAttribute(k2_seq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, K2_SMEM_BYTES);
}

cudaError_t k2_launch_fold(const K2Args &a, cudaStream_t stream)
{
    if (a.S == 0) {
        k2_empty_kernel<<<1, 1, 0, stream>>>(a);
        return cudaGetLastError();
    }
    cudaError_t e = cudaMemsetAsync(a.claim, 0, 256, stream);   // the fold's ticket
    if (e != cudaSuccess)
        return e;
    k2_fold_kernel<<<static_cast<unsigned>(k2_blocks(a.S)), K2_FOLD_THREADS, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t k2_launch(const K2Args &a, int num_sms, cudaStream_t stream)
{
    if (a.S == 0) {
        k2_empty_kernel<<<1, 1, 0, stream>>>(a);
        return cudaGetLastError();
    }
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // the sequence counter and the fold's ticket start at zero
    cudaError_t e = cudaMemsetAsync(a.claim, 0, 256, stream);
    if (e != cudaSuccess)
        return e;
    cfg.gridDim = dim3(std::min(a.S, num_sms * K2_CTAS_PER_SM), 1, 1);
    cfg.blockDim = dim3(K2_THREADS, 1, 1);
    cfg.dynamicSmemBytes = K2_SMEM_BYTES;
    if ((e = cudaLaunchKernelEx(&cfg, k2_seq_kernel, a)) != cudaSuccess)
        return e;
    cfg.gridDim = dim3(static_cast<unsigned>(k2_blocks(a.S)), 1, 1);
    cfg.blockDim = dim3(K2_FOLD_THREADS, 1, 1);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, k2_fold_kernel, a);
}

} // namespace tim
