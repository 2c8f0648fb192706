// tis_ppo.cu -- TIS-weighted PPO clipped surrogate, its gradient and masked means, for sm_103a.
//
// Per token (VeXact summary eq. (2)-(3) with the TIS correction; LoongSage
// "Train-Inference Consistency" section 4; HN page, section on clipped
// importance ratios):
//   r = e^(l_theta - l_old),  w = min(e^(l_old - l_rollout), C),
//   loss = -w min(r A, clip(r, 1 - eps_low, 1 + eps_high) A),
//   grad = -w r A on the unclipped branch, 0 on the clipped one.
// Per sequence: mean loss over its used tokens; per batch: token mean, mean of
// sequence means, clip fractions.
//
// Two launches, fp32 and integer arithmetic only:
//  1. ppo_seq_kernel, three 256-thread CTAs per SM.  A sequence of at most 8192
//     tokens is handled by one warp, a longer one by a whole CTA.  A warp steps
//     through its sequence 256 tokens at a time: lane i owns the tokens at index
//     64 q + i and 64 q + 32 + i (q = 0..3) of the step, loads all of their five
//     inputs first (40 loads in flight per lane, coalesced 128-byte rows per
//     warp), then computes and streams out loss and gradient.  The per-lane
//     loss sums follow the same fixed order as the token indices, a fixed
//     shuffle tree (and for a CTA a warp-ordered sum) gives the sequence total:
//     the order depends only on a token's index inside its own sequence and on
//     the sequence's length, so a sequence's record has the same bits wherever
//     it is packed and whatever else is in the batch.
//     Per token the kernel moves 25 bytes (four fp32 and one byte in, two fp32
//     out), so HBM bounds it; there is no staging and no wait to bound.
//  2. ppo_fold_kernel: CTA j folds sequences 1024 j .. 1024 j + 1023 (4 per
//     thread, structure-of-arrays records) with float-float (TwoSum) sums and
//     integer counts in a fixed tree; when there are several CTAs, the last one
//     to finish folds their partials in index order.
// The batch record depends on S and the sequence records only.
#include <algorithm>
#include <cfloat>

#include "ppo_internal.h"
#include "tim_internal.h"
#include "tim_ptx.cuh"
#include "../../include/tim.h"

namespace tim {
namespace {

// Sequence record, structure of arrays: word f of sequence s is rec[f * S + s].
enum { R_VALID = 0, R_N_MASK, R_N_USED, R_N_PPO, R_N_TIS, R_SUM };
static_assert(R_SUM + 1 == PPO_REC_WORDS, "record layout");

// Fold partial: NCNT int64 counts, NDF float-float sums.
enum { P_N_MASK = 0, P_N_USED, P_N_PPO, P_N_TIS, P_NONEMPTY, P_INVALID, NCNT };
enum { S_LOSS = 0, S_SEQMEAN, NDF };
static_assert(2 * NCNT + 2 * NDF <= PPO_PART_WORDS, "partial layout");

constexpr float kLog2e = 1.4426950408889634f;

// Float-float value hi + lo; addition by Knuth's TwoSum on the high parts with
// the low parts added to the error term, then renormalised.
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

struct PpoAcc {
    float2 inner;   // loss sums of the current step: .x tokens 64 q + lane, .y tokens 64 q + 32 + lane
    float outer;    // the lane's running total over steps
    int n_mask, n_used, n_ppo, n_tis;
};

__device__ __forceinline__ void acc_zero(PpoAcc &t)
{
    t.inner = make_float2(0.f, 0.f);
    t.outer = 0.f;
    t.n_mask = t.n_used = t.n_ppo = t.n_tis = 0;
}

// One token: counts into `t`, returns the loss (0 when not used) and the
// gradient in `grad`.  r is capped at FLT_MAX so that A = 0 gives 0, not NaN.
__device__ __forceinline__ float ppo_token(PpoAcc &t, const PpoArgs &a, float lt, float lo, float lr, float A,
                                           bool m, float &grad)
{
    const float dt = __fsub_rn(lt, lo);
    const float dc = __fsub_rn(lo, lr);
    const bool used = m && fabsf(dt) <= FLT_MAX && fabsf(dc) <= FLT_MAX && fabsf(A) <= FLT_MAX;
    const float r = fminf(ex2(__fmul_rn(dt, kLog2e)), FLT_MAX);
    const float w = fminf(ex2(__fmul_rn(dc, kLog2e)), a.C);
    const bool clip_hi = A > 0.f && dt > a.log_hi_down;
    const bool clip_lo = A < 0.f && dt < a.log_lo_up;
    const bool clipped = clip_hi || clip_lo;
    const float nwA = -(w * A);
    const float unclipped = nwA * r;
    const float loss = clipped ? nwA * (clip_hi ? a.r_hi : a.r_lo) : unclipped;
    grad = used && !clipped ? unclipped : 0.f;
    t.n_mask += static_cast<int>(m);
    t.n_used += static_cast<int>(used);
    t.n_ppo += static_cast<int>(used && clipped);
    t.n_tis += static_cast<int>(used && dc > a.log_c_down);
    return used ? loss : 0.f;
}

// One 256-token step of a sequence: tokens [t0, t0 + n), n <= PPO_CHUNK.  All
// loads are issued before the first use; FULL drops the bounds checks.
template <bool FULL>
__device__ __forceinline__ void ppo_step(PpoAcc &acc, const PpoArgs &a, int64_t t0, int n, int lane)
{
    constexpr int K = PPO_CHUNK / 32;
    float lt[K], lo[K], lr[K], A[K];
    uint8_t m[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int j = 64 * (k >> 1) + 32 * (k & 1) + lane;
        const int64_t t = t0 + j;
        const bool in = FULL || j < n;
        lt[k] = in ? __ldcs(a.l_th + t) : 0.f;
        lo[k] = in ? __ldcs(a.l_old + t) : 0.f;
        lr[k] = in ? __ldcs(a.l_ro + t) : 0.f;
        A[k] = in ? __ldcs(a.adv + t) : 0.f;
        m[k] = in ? __ldcs(a.mask + t) : static_cast<uint8_t>(0);
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int j = 64 * (k >> 1) + 32 * (k & 1) + lane;
        const int64_t t = t0 + j;
        const bool in = FULL || j < n;
        TIM_DCHECK(!in || m[k] <= 1, a.status, TIM_CHECK_MASK, t, m[k]);
        TIM_DCHECK(!in || m[k] == 0 || isfinite(A[k]), a.status, TIM_CHECK_ADVANTAGE, t, __float_as_uint(A[k]));
        float g;
        const float loss = ppo_token(acc, a, lt[k], lo[k], lr[k], A[k], m[k] != 0, g);
        if (k & 1)
            acc.inner.y += loss;
        else
            acc.inner.x += loss;
        if (a.token_loss && in)
            __stcs(a.token_loss + t, loss);
        if (a.token_grad && in)
            __stcs(a.token_grad + t, g);
    }
    acc.outer += acc.inner.x + acc.inner.y;
    acc.inner = make_float2(0.f, 0.f);
}

// L2 prefetch of tokens [t0, t1) of the five input arrays, one bulk prefetch
// per array on lanes 0..4.  Each byte range is widened to whole 16-byte
// granules (the instruction's alignment rule); a granule holding a byte of an
// array lies in a page of that array, so nothing outside the arrays' pages is
// touched.  A prefetch is only a hint: the loads that follow stay correct
// whether or not it has landed.
__device__ __forceinline__ void prefetch_tokens(const PpoArgs &a, int64_t t0, int64_t t1, int lane)
{
    if (lane >= 5 || t1 <= t0)
        return;
    const void *base = lane == 0 ? static_cast<const void *>(a.l_th)
                     : lane == 1 ? static_cast<const void *>(a.l_old)
                     : lane == 2 ? static_cast<const void *>(a.l_ro)
                     : lane == 3 ? static_cast<const void *>(a.adv)
                                 : static_cast<const void *>(a.mask);
    const int64_t esz = lane == 4 ? 1 : 4;
    const uintptr_t lo = (reinterpret_cast<uintptr_t>(base) + t0 * esz) & ~uintptr_t(15);
    const uintptr_t hi = (reinterpret_cast<uintptr_t>(base) + t1 * esz + 15) & ~uintptr_t(15);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                 :: "l"(lo), "r"(static_cast<uint32_t>(hi - lo)) : "memory");
}

__device__ __forceinline__ void ppo_range(PpoAcc &acc, const PpoArgs &a, int64_t t0, int64_t e, int lane)
{
    if (e - t0 >= PPO_CHUNK)
        ppo_step<true>(acc, a, t0, PPO_CHUNK, lane);
    else
        ppo_step<false>(acc, a, t0, static_cast<int>(e - t0), lane);
}

struct SeqTot {
    float sum;
    int cnt[4];   // n_mask, n_used, n_ppo, n_tis
};

// Fixed xor-shuffle tree over a warp; the sum is taken from lane 0 and
// broadcast, so every lane holds the same bits.
__device__ __forceinline__ SeqTot warp_total(const PpoAcc &acc)
{
    SeqTot t;
    t.sum = acc.outer;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        t.sum += __shfl_xor_sync(0xffffffffu, t.sum, o);
    t.sum = __shfl_sync(0xffffffffu, t.sum, 0);
    t.cnt[0] = __reduce_add_sync(0xffffffffu, acc.n_mask);
    t.cnt[1] = __reduce_add_sync(0xffffffffu, acc.n_used);
    t.cnt[2] = __reduce_add_sync(0xffffffffu, acc.n_ppo);
    t.cnt[3] = __reduce_add_sync(0xffffffffu, acc.n_tis);
    return t;
}

// Output and workspace record of sequence s, by one full warp whose lanes
// hold the same totals (lane i writes record word i).
__device__ __forceinline__ void write_seq(const PpoArgs &a, int s, const SeqTot &t, int lane)
{
    const size_t S = static_cast<size_t>(a.S);
    if (lane == 0)
        a.seq_loss[s] = t.cnt[1] > 0 ? __fdiv_rn(t.sum, static_cast<float>(t.cnt[1])) : 0.f;
    uint32_t v = 1u;   // R_VALID
    v = lane == R_N_MASK ? static_cast<uint32_t>(t.cnt[0]) : v;
    v = lane == R_N_USED ? static_cast<uint32_t>(t.cnt[1]) : v;
    v = lane == R_N_PPO ? static_cast<uint32_t>(t.cnt[2]) : v;
    v = lane == R_N_TIS ? static_cast<uint32_t>(t.cnt[3]) : v;
    v = lane == R_SUM ? __float_as_uint(t.sum) : v;
    if (lane < PPO_REC_WORDS)
        a.rec[lane * S + s] = v;
}

__device__ __forceinline__ bool offsets_ok(const PpoArgs &a, int s, int64_t b, int64_t e)
{
    bool ok = b >= 0 && e >= b && e <= a.N;
    if (s == 0 && b != 0)
        ok = false;
    if (s == a.S - 1 && e != a.N)
        ok = false;
    return ok;
}

// Record of a sequence that is not stepped through: bad offsets (NaN mean,
// invalid record, status) or no tokens (all zero).
__device__ __forceinline__ void write_plain(const PpoArgs &a, int s, bool bad, int lane)
{
    if (bad) {
        if (lane == 0) {
            atomicCAS(a.status, 0, static_cast<int>(TIM_ERR_BAD_INPUT));
            a.seq_loss[s] = qnan();
        }
        if (lane < PPO_REC_WORDS)
            a.rec[static_cast<size_t>(lane) * a.S + s] = 0u;
    } else {
        SeqTot z;
        z.sum = 0.f;
        z.cnt[0] = z.cnt[1] = z.cnt[2] = z.cnt[3] = 0;
        write_seq(a, s, z, lane);
    }
}

__global__ void __launch_bounds__(PPO_THREADS, PPO_CTAS_PER_SM) ppo_seq_kernel(const PpoArgs a)
{
    __shared__ float red_f[PPO_WARPS];
    __shared__ int red_i[PPO_WARPS][4];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();                // the inputs may be written by the previous kernel
    pdl_launch_dependents();   // the fold kernel may start launching
    if (blockIdx.x == 0 && tid == 0)
        *a.ticket = 0u;        // the fold kernel reads it after this grid completes
    bool mine = false;         // does this CTA own a sequence longer than PPO_LONG?
    for (int q = blockIdx.x + tid * gridDim.x; q < a.S; q += PPO_THREADS * gridDim.x) {
        const int64_t b = a.off[q], e = a.off[q + 1];
        mine = mine || (offsets_ok(a, q, b, e) && e - b > PPO_LONG);
    }
    const bool has_long = __syncthreads_or(mine) != 0;

    // ---- phase 1: sequences of at most PPO_LONG tokens, one warp each.  Warps
    // claim tickets in index order from the call's counter, one ticket ahead of
    // the range they reduce: in a large batch the first tickets hand out
    // PPO_CLAIM_BLOCK consecutive sequences each (few claims on the counter's
    // word), the last ones, and every ticket of a batch of at most two
    // sequences per warp, one sequence each.  Which warp handles a sequence
    // never changes its record's bits.  Each sequence is prefetched into L2
    // ahead of the warp's loads: its first two steps when it starts, step c + 2
    // during step c.  (Prefetching the warp's next sequence as well was
    // measured slower: ~20% of it was fetched from DRAM twice.)
    const int singles = min(a.S, max(a.S / 8, 2 * static_cast<int>(gridDim.x) * PPO_WARPS));
    const int t_blocks = (a.S - singles) / PPO_CLAIM_BLOCK;   // tickets of PPO_CLAIM_BLOCK sequences
    int pend = lane == 0 ? atomicAdd(a.claim, 1) : 0;       // lane 0: the next ticket
    int t_cur = 0, t_end = 0;                               // the current ticket's sequences
    while (true) {
        if (t_cur >= t_end) {
            const int t = __shfl_sync(0xffffffffu, pend, 0);
            pend = lane == 0 ? atomicAdd(a.claim, 1) : 0;
            if (t < t_blocks) {
                t_cur = t * PPO_CLAIM_BLOCK;
                t_end = t_cur + PPO_CLAIM_BLOCK;
            } else {
                t_cur = t_blocks * PPO_CLAIM_BLOCK + (t - t_blocks);   // t < S + claims in flight: no overflow
                t_end = t_cur + 1;
            }
            if (t_cur >= a.S)   // every later ticket is past S too
                break;
            t_end = min(t_end, a.S);
        }
        const int s = t_cur++;
        const int64_t b = a.off[s], e = a.off[s + 1];
        if (!offsets_ok(a, s, b, e)) {
            write_plain(a, s, true, lane);
            continue;
        }
        if (e - b > PPO_LONG)
            continue;
        prefetch_tokens(a, b, min(e, b + 2 * PPO_CHUNK), lane);
        PpoAcc acc;
        acc_zero(acc);
        for (int64_t t0 = b; t0 < e; t0 += PPO_CHUNK) {
            prefetch_tokens(a, t0 + 2 * PPO_CHUNK, min(e, t0 + 3 * PPO_CHUNK), lane);
            ppo_range(acc, a, t0, e, lane);
        }
        write_seq(a, s, warp_total(acc), lane);
    }

    // ---- phase 2: longer sequences, one CTA each (q = blockIdx.x + k gridDim.x, as
    // the pre-scan above); warp w takes steps w, w + PPO_WARPS, ...
    if (!has_long)   // uniform over the CTA
        return;
    for (int q = blockIdx.x; q < a.S; q += gridDim.x) {
        const int64_t b = a.off[q], e = a.off[q + 1];
        if (!offsets_ok(a, q, b, e) || e - b <= PPO_LONG)   // uniform over the CTA
            continue;
        __syncthreads();   // the previous long sequence's reduction buffers are free
        PpoAcc acc;
        acc_zero(acc);
        for (int64_t t0 = b + static_cast<int64_t>(warp) * PPO_CHUNK; t0 < e; t0 += PPO_WARPS * PPO_CHUNK) {
            const int64_t p0 = t0 + PPO_WARPS * PPO_CHUNK;   // this warp's next step
            prefetch_tokens(a, p0, min(e, p0 + PPO_CHUNK), lane);
            ppo_range(acc, a, t0, e, lane);
        }
        const SeqTot t = warp_total(acc);
        if (lane == 0) {
            red_f[warp] = t.sum;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                red_i[warp][k] = t.cnt[k];
        }
        __syncthreads();
        if (warp == 0) {   // every lane folds the warps in order: the same bits on all lanes
            SeqTot c;
            c.sum = 0.f;
            c.cnt[0] = c.cnt[1] = c.cnt[2] = c.cnt[3] = 0;
            for (int w = 0; w < PPO_WARPS; ++w) {
                c.sum += red_f[w];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    c.cnt[k] += red_i[w][k];
            }
            write_seq(a, q, c, lane);
        }
    }
}

struct FoldAcc {
    long long cnt[NCNT];
    ff sum[NDF];
};

__device__ __forceinline__ void fold_zero(FoldAcc &f)
{
#pragma unroll
    for (int i = 0; i < NCNT; ++i)
        f.cnt[i] = 0;
#pragma unroll
    for (int i = 0; i < NDF; ++i)
        f.sum[i] = {0.f, 0.f};
}

__device__ __forceinline__ void fold_add(FoldAcc &x, const FoldAcc &y)
{
#pragma unroll
    for (int i = 0; i < NCNT; ++i)
        x.cnt[i] += y.cnt[i];
#pragma unroll
    for (int i = 0; i < NDF; ++i)
        x.sum[i] = ff_add(x.sum[i], y.sum[i]);
}

__device__ __forceinline__ FoldAcc fold_shfl_xor(const FoldAcc &x, int o)
{
    FoldAcc y;
#pragma unroll
    for (int i = 0; i < NCNT; ++i)
        y.cnt[i] = __shfl_xor_sync(0xffffffffu, x.cnt[i], o);
#pragma unroll
    for (int i = 0; i < NDF; ++i) {
        y.sum[i].hi = __shfl_xor_sync(0xffffffffu, x.sum[i].hi, o);
        y.sum[i].lo = __shfl_xor_sync(0xffffffffu, x.sum[i].lo, o);
    }
    return y;
}

__device__ __forceinline__ void fold_store(uint32_t *p, const FoldAcc &f)
{
    for (int i = 0; i < NCNT; ++i) {
        p[2 * i] = static_cast<uint32_t>(static_cast<unsigned long long>(f.cnt[i]));
        p[2 * i + 1] = static_cast<uint32_t>(static_cast<unsigned long long>(f.cnt[i]) >> 32);
    }
    for (int i = 0; i < NDF; ++i) {
        p[2 * NCNT + 2 * i] = __float_as_uint(f.sum[i].hi);
        p[2 * NCNT + 2 * i + 1] = __float_as_uint(f.sum[i].lo);
    }
}

__device__ __forceinline__ void fold_load(FoldAcc &f, const uint32_t *p)
{
#pragma unroll
    for (int i = 0; i < NCNT; ++i)
        f.cnt[i] = static_cast<long long>(static_cast<unsigned long long>(p[2 * i]) |
                                          (static_cast<unsigned long long>(p[2 * i + 1]) << 32));
#pragma unroll
    for (int i = 0; i < NDF; ++i)
        f.sum[i] = {__uint_as_float(p[2 * NCNT + 2 * i]), __uint_as_float(p[2 * NCNT + 2 * i + 1])};
}

// Fixed tree over a CTA: xor shuffles inside each warp, then the same over the
// warp totals in warp 0.  Returns the total on thread 0.
__device__ __forceinline__ FoldAcc fold_cta(FoldAcc x)
{
    constexpr int NW = PPO_FOLD_THREADS / 32;
    static_assert((NW & (NW - 1)) == 0 && NW <= 32, "warps per fold CTA");
    __shared__ uint32_t sh[NW][PPO_PART_WORDS];
#pragma unroll 1
    for (int o = 16; o > 0; o >>= 1)
        fold_add(x, fold_shfl_xor(x, o));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0)
        fold_store(sh[warp], x);
    __syncthreads();
    FoldAcc t;
    fold_zero(t);
    if (warp == 0) {
        if (lane < NW)
            fold_load(t, sh[lane]);
#pragma unroll 1
        for (int o = NW / 2; o > 0; o >>= 1)
            fold_add(t, fold_shfl_xor(t, o));
    }
    return t;
}

// fp32 -> fp64 by moving bits (exact; fp32 subnormals renormalised), so that
// the batch record needs no fp64 arithmetic.
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

// A count (< 2^53) as fp64, by moving bits.
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
// fp32 quotients of the float-float sums and the counts.
__device__ void write_batch(const PpoArgs &a, const FoldAcc &t, bool check_offsets)
{
    bool bad = t.cnt[P_INVALID] > 0;
    if (check_offsets)
        bad = bad || a.off[0] != 0 || static_cast<int64_t>(a.off[a.S]) != a.N;
    if (bad)
        atomicCAS(a.status, 0, static_cast<int>(TIM_ERR_BAD_INPUT));
    const float n_used = static_cast<float>(t.cnt[P_N_USED]);
    const float n_ne = static_cast<float>(t.cnt[P_NONEMPTY]);
    auto mean = [&](int i, float n) { return n > 0.f ? widen((t.sum[i].hi + t.sum[i].lo) / n) : 0.0; };
    auto ratio = [](long long x, float n) { return n > 0.f ? widen(static_cast<float>(x) / n) : 0.0; };
    double *o = a.batch;
    o[TIM_PPO_N_MASK] = widen_count(t.cnt[P_N_MASK]);
    o[TIM_PPO_N_USED] = widen_count(t.cnt[P_N_USED]);
    o[TIM_PPO_N_PPO_CLIPPED] = widen_count(t.cnt[P_N_PPO]);
    o[TIM_PPO_N_TIS_CLIPPED] = widen_count(t.cnt[P_N_TIS]);
    o[TIM_PPO_MEAN_LOSS] = mean(S_LOSS, n_used);
    o[TIM_PPO_SEQMEAN_LOSS] = mean(S_SEQMEAN, n_ne);
    o[TIM_PPO_PPO_CLIP_RATIO] = ratio(t.cnt[P_N_PPO], n_used);
    o[TIM_PPO_TIS_CLIP_RATIO] = ratio(t.cnt[P_N_TIS], n_used);
    o[TIM_PPO_N_SEQS_NONEMPTY] = widen_count(t.cnt[P_NONEMPTY]);
    if (bad)
        for (int f = 0; f < TIM_PPO_FIELDS; ++f)
            o[f] = __longlong_as_double(0x7ff8000000000000ll);
}

// The fold term of sequence s.
// The words of sequence s that the fold reads: its record and its mean.  Every
// sequence has both (a bad one an all-zero record), so they are loaded
// unconditionally, all sequences of a thread at once.
struct SeqWords {
    uint32_t w[PPO_REC_WORDS];
    float mean;
};

__device__ __forceinline__ SeqWords load_seq(const PpoArgs &a, int64_t s)
{
    const size_t S = static_cast<size_t>(a.S);
    SeqWords v;
#pragma unroll
    for (int f = 0; f < PPO_REC_WORDS; ++f)
        v.w[f] = __ldg(a.rec + f * S + s);
    v.mean = __ldg(a.seq_loss + s);
    return v;
}

// The fold term of one sequence.
__device__ __forceinline__ void fold_seq(FoldAcc &x, const SeqWords &v)
{
    FoldAcc y;
    fold_zero(y);
    if (v.w[R_VALID] == 0u) {
        y.cnt[P_INVALID] = 1;
    } else {
        const uint32_t nu = v.w[R_N_USED];
        y.cnt[P_N_MASK] = v.w[R_N_MASK];
        y.cnt[P_N_USED] = nu;
        y.cnt[P_N_PPO] = v.w[R_N_PPO];
        y.cnt[P_N_TIS] = v.w[R_N_TIS];
        y.sum[S_LOSS] = {__uint_as_float(v.w[R_SUM]), 0.f};
        if (nu > 0u) {
            y.cnt[P_NONEMPTY] = 1;
            y.sum[S_SEQMEAN] = {v.mean, 0.f};
        }
    }
    fold_add(x, y);
}

// CTA j folds sequences 1024 j + i + 256 k (k = 0..3, in order) on thread i.
// With a single CTA it writes the batch record directly; otherwise each CTA
// stores its partial and the CTA that finishes last (a ticket counter) folds
// the partials in index order, thread i taking partials i, i + 256, ...  The
// result does not depend on which CTA finishes last.
__global__ void __launch_bounds__(PPO_FOLD_THREADS) ppo_fold_kernel(const PpoArgs a)
{
    __shared__ int last_s;
    pdl_wait();   // the records (and the zeroed ticket) come from ppo_seq_kernel
    pdl_launch_dependents();
    FoldAcc x;
    fold_zero(x);
    const int64_t base = static_cast<int64_t>(blockIdx.x) * PPO_FOLD_SEQS + threadIdx.x;
    constexpr int KS = PPO_FOLD_SEQS / PPO_FOLD_THREADS;
    SeqWords v[KS];
#pragma unroll
    for (int k = 0; k < KS; ++k) {
        const int64_t s = base + static_cast<int64_t>(k) * PPO_FOLD_THREADS;
        if (s < a.S)
            v[k] = load_seq(a, s);
    }
#pragma unroll
    for (int k = 0; k < KS; ++k)
        if (base + static_cast<int64_t>(k) * PPO_FOLD_THREADS < a.S)
            fold_seq(x, v[k]);
    const FoldAcc t = fold_cta(x);
    if (threadIdx.x == 0) {
        if (gridDim.x == 1) {
            write_batch(a, t, false);
        } else {
            fold_store(a.part + static_cast<size_t>(blockIdx.x) * PPO_PART_WORDS, t);
            __threadfence();
            last_s = atomicAdd(a.ticket, 1u) == gridDim.x - 1;
        }
    }
    if (gridDim.x == 1)
        return;
    __syncthreads();
    if (!last_s)   // uniform over the CTA
        return;
    __threadfence();
    FoldAcc y;
    fold_zero(y);
    for (int p = threadIdx.x; p < static_cast<int>(gridDim.x); p += PPO_FOLD_THREADS) {
        const uint32_t *src = a.part + static_cast<size_t>(p) * PPO_PART_WORDS;
        uint32_t w[PPO_PART_WORDS];
#pragma unroll
        for (int i = 0; i < PPO_PART_WORDS; ++i)
            w[i] = __ldcg(src + i);   // written by other CTAs: read through L2
        FoldAcc z;
        fold_load(z, w);
        fold_add(y, z);
    }
    const FoldAcc f = fold_cta(y);
    if (threadIdx.x == 0)
        write_batch(a, f, false);
}

// S = 0: only the (all-zero) batch record, after checking the offsets cover [0, N).
__global__ void ppo_empty_kernel(const PpoArgs a)
{
    FoldAcc t;
    fold_zero(t);
    write_batch(a, t, true);
}

} // namespace

cudaError_t ppo_launch(const PpoArgs &a, int num_sms, cudaStream_t stream)
{
    if (a.S == 0) {
        ppo_empty_kernel<<<1, 1, 0, stream>>>(a);
        return cudaGetLastError();
    }
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(std::min(a.S, num_sms * PPO_CTAS_PER_SM), 1, 1);
    cfg.blockDim = dim3(PPO_THREADS, 1, 1);
    cudaError_t e = cudaMemsetAsync(a.claim, 0, sizeof(int), stream);
    if (e == cudaSuccess)
        e = cudaLaunchKernelEx(&cfg, ppo_seq_kernel, a);
    if (e != cudaSuccess)
        return e;
    const int parts = (a.S + PPO_FOLD_SEQS - 1) / PPO_FOLD_SEQS;
    cfg.gridDim = dim3(parts, 1, 1);
    cfg.blockDim = dim3(PPO_FOLD_THREADS, 1, 1);
    return cudaLaunchKernelEx(&cfg, ppo_fold_kernel, a);
}

} // namespace tim
