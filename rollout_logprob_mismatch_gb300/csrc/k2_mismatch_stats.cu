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
// One CTA reduces one sequence at a time (grid-stride over sequences).  Thread i
// owns the tokens whose index inside the sequence is i, i + 256, i + 512, ...,
// sums them in that order (fp32, folded every 16 rounds into a compensated
// fp32 total), then a fixed shuffle tree and a warp-ordered fp64 sum give the
// sequence totals.  The order depends only on a token's index inside its own
// sequence, so a sequence's record is bit-identical wherever it is packed and
// whatever else is in the batch.  A single CTA then folds the sequence records
// in index order (fp64) into the batch record.
#include <algorithm>
#include <cfloat>

#include "tim_internal.h"
#include "../../include/tim.h"

namespace tim {
namespace {

enum { F_D = 0, F_AD, F_K2, F_K3, F_W, F_REL, NSUM };

// Workspace record of one sequence (doubles).
enum {
    R_VALID = 0, R_N_MASK, R_N_USED, R_N_NAN, R_N_CLIP, R_SD, R_SAD, R_SK2, R_SK3, R_SW, R_SREL,
    R_MAX, R_MK1, R_MK2, R_MK3, R_FLAG
};
static_assert(R_FLAG + 1 == K2_REC, "record layout");

// e^d - 1 - d.  For |d| < 0.5 the Taylor series sum_{n>=2} d^n / n! through n = 9
// (truncation below 2e-9 relative); above, expm1f(d) - d loses no digits.
__device__ __forceinline__ float k3_of(float d)
{
    if (fabsf(d) < 0.5f) {
        float p = 1.f / 362880.f;
        p = fmaf(p, d, 1.f / 40320.f);
        p = fmaf(p, d, 1.f / 5040.f);
        p = fmaf(p, d, 1.f / 720.f);
        p = fmaf(p, d, 1.f / 120.f);
        p = fmaf(p, d, 1.f / 24.f);
        p = fmaf(p, d, 1.f / 6.f);
        p = fmaf(p, d, 0.5f);
        return d * d * p;
    }
    return expm1f(d) - d;
}

// Neumaier's compensated addition of x into (sum, comp).
__device__ __forceinline__ void neumaier(float &sum, float &comp, float x)
{
    const float t = sum + x;
    if (fabsf(sum) >= fabsf(x))
        comp += (sum - t) + x;
    else
        comp += (x - t) + sum;
    sum = t;
}

__device__ __forceinline__ float qnan() { return __int_as_float(0x7fc00000); }

__global__ void __launch_bounds__(K2_THREADS) k2_seq_kernel(const K2Args a)
{
    constexpr int NW = K2_THREADS / 32;
    __shared__ float red_f[NW][NSUM];
    __shared__ int red_i[NW][4];
    __shared__ float red_mx[NW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int s = blockIdx.x; s < a.S; s += gridDim.x) {
        const int64_t b = a.off[s], e = a.off[s + 1];
        bool valid = b >= 0 && e >= b && e <= a.N;
        if (s == 0 && b != 0)
            valid = false;
        if (s == a.S - 1 && e != a.N)
            valid = false;
        if (!valid) {   // uniform over the CTA: every thread read the same offsets
            if (tid == 0) {
                atomicCAS(a.status, 0, static_cast<int>(TIM_ERR_BAD_INPUT));
                for (int f = 0; f < TIM_SEQ_FIELDS; ++f)
                    a.seq_stats[static_cast<size_t>(s) * TIM_SEQ_FIELDS + f] = qnan();
                a.seq_flags[s] = 0;
                for (int f = 0; f < K2_REC; ++f)
                    a.rec[static_cast<size_t>(s) * K2_REC + f] = 0.0;
            }
            continue;
        }
        const int64_t len = e - b;
        const int64_t nrounds = (len + K2_THREADS - 1) / K2_THREADS;
        float outer[NSUM], comp[NSUM];
#pragma unroll
        for (int f = 0; f < NSUM; ++f)
            outer[f] = comp[f] = 0.f;
        float mx = 0.f;
        int n_mask = 0, n_used = 0, n_nan = 0, n_clip = 0;

        for (int64_t r0 = 0; r0 < nrounds; r0 += K2_GROUP) {
            const int64_t r1 = min(nrounds, r0 + static_cast<int64_t>(K2_GROUP));
            float inner[NSUM];
#pragma unroll
            for (int f = 0; f < NSUM; ++f)
                inner[f] = 0.f;
            for (int64_t r = r0; r < r1; r += 4) {
                float lt[4], lr[4];
                uint32_t mk[4];
                bool in[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int64_t rel = (r + k) * K2_THREADS + tid;
                    in[k] = (r + k < r1) && (rel < len);
                    const int64_t t = b + rel;
                    lt[k] = in[k] ? __ldcs(a.l_tr + t) : 0.f;
                    lr[k] = in[k] ? __ldcs(a.l_ro + t) : 0.f;
                    mk[k] = in[k] ? static_cast<uint32_t>(__ldcs(a.mask + t)) : 0u;
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (!in[k])
                        continue;
                    const bool m = mk[k] != 0u;
                    const float d = lt[k] - lr[k];
                    const bool fin = fabsf(d) <= FLT_MAX;   // false for inf and NaN
                    n_mask += m;
                    n_nan += m && !fin;
                    float w = 0.f;
                    if (m && fin) {
                        const float r_ = expf(d);
                        const float ad = fabsf(d);
                        w = fminf(r_, a.C);
                        n_used += 1;
                        n_clip += d > a.log_c_down;
                        inner[F_D] += d;
                        inner[F_AD] += ad;
                        inner[F_K2] += 0.5f * d * d;
                        inner[F_K3] += k3_of(d);
                        inner[F_W] += w;
                        inner[F_REL] += ad / (fabsf(lt[k]) + 1e-8f);
                        mx = fmaxf(mx, ad);
                    }
                    if (a.token_weight)
                        a.token_weight[b + (r + k) * K2_THREADS + tid] = w;
                }
            }
#pragma unroll
            for (int f = 0; f < NSUM; ++f)
                neumaier(outer[f], comp[f], inner[f]);
        }

        float tot[NSUM];
#pragma unroll
        for (int f = 0; f < NSUM; ++f) {
            tot[f] = outer[f] + comp[f];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                tot[f] += __shfl_xor_sync(0xffffffffu, tot[f], o);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        n_mask = __reduce_add_sync(0xffffffffu, n_mask);
        n_used = __reduce_add_sync(0xffffffffu, n_used);
        n_nan = __reduce_add_sync(0xffffffffu, n_nan);
        n_clip = __reduce_add_sync(0xffffffffu, n_clip);
        if (lane == 0) {
#pragma unroll
            for (int f = 0; f < NSUM; ++f)
                red_f[warp][f] = tot[f];
            red_i[warp][0] = n_mask;
            red_i[warp][1] = n_used;
            red_i[warp][2] = n_nan;
            red_i[warp][3] = n_clip;
            red_mx[warp] = mx;
        }
        __syncthreads();
        if (tid == 0) {
            double sum[NSUM] = {0, 0, 0, 0, 0, 0};
            long long cnt[4] = {0, 0, 0, 0};
            float m = 0.f;
            for (int w = 0; w < NW; ++w) {
                for (int f = 0; f < NSUM; ++f)
                    sum[f] += static_cast<double>(red_f[w][f]);
                for (int c = 0; c < 4; ++c)
                    cnt[c] += red_i[w][c];
                m = fmaxf(m, red_mx[w]);
            }
            const double nu = static_cast<double>(cnt[1]);
            auto mean = [&](double x) { return cnt[1] > 0 ? x / nu : 0.0; };
            const double md = mean(sum[F_D]);
            const double mk1 = -md;
            const double mk2 = mean(sum[F_K2]);
            const double mk3 = mean(sum[F_K3]);
            float *o = a.seq_stats + static_cast<size_t>(s) * TIM_SEQ_FIELDS;
            o[TIM_SEQ_N_MASK] = static_cast<float>(cnt[0]);
            o[TIM_SEQ_N_USED] = static_cast<float>(cnt[1]);
            o[TIM_SEQ_N_NAN] = static_cast<float>(cnt[2]);
            o[TIM_SEQ_N_CLIP] = static_cast<float>(cnt[3]);
            o[TIM_SEQ_MEAN_DELTA] = static_cast<float>(md);
            o[TIM_SEQ_MEAN_ABS_DELTA] = static_cast<float>(mean(sum[F_AD]));
            o[TIM_SEQ_MAX_ABS_DELTA] = m;
            o[TIM_SEQ_MEAN_K1] = static_cast<float>(mk1);
            o[TIM_SEQ_MEAN_K2] = static_cast<float>(mk2);
            o[TIM_SEQ_MEAN_K3] = static_cast<float>(mk3);
            o[TIM_SEQ_MEAN_W] = static_cast<float>(mean(sum[F_W]));
            o[TIM_SEQ_MEAN_REL] = static_cast<float>(mean(sum[F_REL]));
            int flag = 0;
            if (cnt[1] > 0)
                flag = (a.estimator == 3 ? mk3 : fabs(mk1)) > a.tau;
            a.seq_flags[s] = flag;
            double *rc = a.rec + static_cast<size_t>(s) * K2_REC;
            rc[R_VALID] = 1.0;
            rc[R_N_MASK] = static_cast<double>(cnt[0]);
            rc[R_N_USED] = nu;
            rc[R_N_NAN] = static_cast<double>(cnt[2]);
            rc[R_N_CLIP] = static_cast<double>(cnt[3]);
            rc[R_SD] = sum[F_D];
            rc[R_SAD] = sum[F_AD];
            rc[R_SK2] = sum[F_K2];
            rc[R_SK3] = sum[F_K3];
            rc[R_SW] = sum[F_W];
            rc[R_SREL] = sum[F_REL];
            rc[R_MAX] = static_cast<double>(m);
            rc[R_MK1] = mk1;
            rc[R_MK2] = mk2;
            rc[R_MK3] = mk3;
            rc[R_FLAG] = static_cast<double>(flag);
        }
        __syncthreads();
    }
}

// Batch record from the sequence records: thread t folds a contiguous slice of
// sequences in index order (fp64), then a fixed shuffle tree and a warp-ordered
// sum finish it.  The result depends on S and the records only.
__global__ void __launch_bounds__(K2_BATCH_THREADS) k2_batch_kernel(const K2Args a)
{
    enum { B_MASK = 0, B_USED, B_NAN, B_CLIP, B_SD, B_SAD, B_SK2, B_SK3, B_SW, B_SREL, B_MK1,
           B_MK2, B_MK3, B_NONEMPTY, B_REJ, B_INVALID, NB };
    constexpr int NW = K2_BATCH_THREADS / 32;
    __shared__ double red[NW][NB];
    __shared__ double red_mx[NW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    double acc[NB];
#pragma unroll
    for (int f = 0; f < NB; ++f)
        acc[f] = 0.0;
    double mx = 0.0;
    const int64_t s_lo = static_cast<int64_t>(a.S) * tid / K2_BATCH_THREADS;
    const int64_t s_hi = static_cast<int64_t>(a.S) * (tid + 1) / K2_BATCH_THREADS;
    for (int64_t s = s_lo; s < s_hi; ++s) {
        const double *rc = a.rec + s * K2_REC;
        if (rc[R_VALID] == 0.0) {
            acc[B_INVALID] += 1.0;
            continue;
        }
        acc[B_MASK] += rc[R_N_MASK];
        acc[B_USED] += rc[R_N_USED];
        acc[B_NAN] += rc[R_N_NAN];
        acc[B_CLIP] += rc[R_N_CLIP];
        acc[B_SD] += rc[R_SD];
        acc[B_SAD] += rc[R_SAD];
        acc[B_SK2] += rc[R_SK2];
        acc[B_SK3] += rc[R_SK3];
        acc[B_SW] += rc[R_SW];
        acc[B_SREL] += rc[R_SREL];
        mx = fmax(mx, rc[R_MAX]);
        if (rc[R_N_USED] > 0.0) {
            acc[B_MK1] += rc[R_MK1];
            acc[B_MK2] += rc[R_MK2];
            acc[B_MK3] += rc[R_MK3];
            acc[B_NONEMPTY] += 1.0;
            acc[B_REJ] += rc[R_FLAG];
        }
    }
#pragma unroll
    for (int f = 0; f < NB; ++f)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            acc[f] += __shfl_xor_sync(0xffffffffu, acc[f], o);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) {
        for (int f = 0; f < NB; ++f)
            red[warp][f] = acc[f];
        red_mx[warp] = mx;
    }
    __syncthreads();
    if (tid != 0)
        return;
    double t[NB];
    for (int f = 0; f < NB; ++f)
        t[f] = 0.0;
    double m = 0.0;
    for (int w = 0; w < NW; ++w) {
        for (int f = 0; f < NB; ++f)
            t[f] += red[w][f];
        m = fmax(m, red_mx[w]);
    }
    // the offsets must cover exactly [0, N); a sequence kernel that found a bad
    // sequence left its record invalid
    const bool bad = t[B_INVALID] > 0.0 || a.off[0] != 0 || static_cast<int64_t>(a.off[a.S]) != a.N;
    if (bad)
        atomicCAS(a.status, 0, static_cast<int>(TIM_ERR_BAD_INPUT));
    auto div = [](double x, double n) { return n > 0.0 ? x / n : 0.0; };
    double *o = a.batch;
    o[TIM_BATCH_N_MASK] = t[B_MASK];
    o[TIM_BATCH_N_USED] = t[B_USED];
    o[TIM_BATCH_N_NAN] = t[B_NAN];
    o[TIM_BATCH_N_CLIP] = t[B_CLIP];
    o[TIM_BATCH_MEAN_DELTA] = div(t[B_SD], t[B_USED]);
    o[TIM_BATCH_MEAN_ABS_DELTA] = div(t[B_SAD], t[B_USED]);
    o[TIM_BATCH_MAX_ABS_DELTA] = m;
    o[TIM_BATCH_MEAN_K1] = -div(t[B_SD], t[B_USED]);
    o[TIM_BATCH_MEAN_K2] = div(t[B_SK2], t[B_USED]);
    o[TIM_BATCH_MEAN_K3] = div(t[B_SK3], t[B_USED]);
    o[TIM_BATCH_MEAN_W] = div(t[B_SW], t[B_USED]);
    o[TIM_BATCH_MEAN_REL] = div(t[B_SREL], t[B_USED]);
    o[TIM_BATCH_SEQMEAN_K1] = div(t[B_MK1], t[B_NONEMPTY]);
    o[TIM_BATCH_SEQMEAN_K2] = div(t[B_MK2], t[B_NONEMPTY]);
    o[TIM_BATCH_SEQMEAN_K3] = div(t[B_MK3], t[B_NONEMPTY]);
    o[TIM_BATCH_CLIP_RATIO] = div(t[B_CLIP], t[B_MASK]);
    o[TIM_BATCH_NAN_RATIO] = div(t[B_NAN], t[B_MASK]);
    o[TIM_BATCH_REJECT_RATIO] = div(t[B_REJ], t[B_NONEMPTY]);
    o[TIM_BATCH_N_SEQS_NONEMPTY] = t[B_NONEMPTY];
    o[TIM_BATCH_N_REJECTED] = t[B_REJ];
    if (bad)
        for (int f = 0; f < TIM_BATCH_FIELDS; ++f)
            o[f] = __longlong_as_double(0x7ff8000000000000ll);
}

} // namespace

cudaError_t k2_launch(const K2Args &a, int num_sms, cudaStream_t stream)
{
    if (a.S > 0) {
        const int grid = static_cast<int>(std::min<int64_t>(a.S, static_cast<int64_t>(num_sms) * 8));
        k2_seq_kernel<<<grid, K2_THREADS, 0, stream>>>(a);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }
    k2_batch_kernel<<<1, K2_BATCH_THREADS, 0, stream>>>(a);
    return cudaGetLastError();
}

} // namespace tim
