// mismatch_monitor.cu -- distribution monitor of the train/rollout mismatch, for sm_103a.
//
// Over the used tokens of a batch (mask != 0, finite fp32 delta = l_train -
// l_rollout): the p95 of |delta|, the 0.01 / 0.5 / 0.99 quantiles of the ratio
// r = e^delta, the count and fraction of tokens with |delta| > tau_tok and the
// per-token rejection flag (llm-infra-atlas "训推一致性与 determinism" section 7,
// the per-token mismatch metrics; VeXact summary, the token threshold tau_tok).
// A quantile at level q is the linear interpolation at h = (n - 1) q between
// the order statistics floor(h) and floor(h) + 1; e^x is increasing, so the
// ratio's order statistics are e^ of delta's.
//
// The eight order statistics (two per quantile) are found exactly, by radix
// selection on 32-bit keys that order like the values (|delta|: its bits;
// delta: sign-flipped bits), in three passes over the tokens of 11, 11 and 10
// key bits:
//   mon_pass_kernel<1>   histogram of the top 11 bits of delta's key (that of
//                        |delta| follows from it), n_used, n_extreme and the
//                        rejection flags;
//   mon_select_kernel<1> ranks from n_used; per target, the bin that holds
//                        its rank and the rank left inside that bin;
//   mon_pass_kernel<2>   per target, histogram of bits 20..10 of the keys in
//                        its bin;  mon_select_kernel<2>;
//   mon_pass_kernel<3>   bits 9..0;  mon_select_kernel<3> ends with exact
//                        keys and writes the record.
// Counts are integers, so the result does not depend on the order in which
// threads add them: the selected tokens are exactly the oracle's.  Each pass
// reads 9 bytes per token; a CTA counts into shared-memory histograms and adds
// the non-zero bins to the global ones at the end.
#include <algorithm>
#include <cfloat>
#include <cmath>

#include "monitor_internal.h"
#include "tim_internal.h"
#include "tim_ptx.cuh"
#include "../../include/tim.h"

namespace tim {
namespace {

// Quantile levels: |delta| at 0.95 (targets 0, 1), the ratio at 0.01, 0.5, 0.99.
__device__ __forceinline__ double level(int i)
{
    return i == 0 ? 0.95 : i == 1 ? 0.01 : i == 2 ? 0.5 : 0.99;
}

// Key of |delta| (targets 0, 1) and of delta (targets 2..7).
__device__ __forceinline__ uint32_t key_abs(float d) { return __float_as_uint(fabsf(d)); }

__device__ __forceinline__ uint32_t key_signed(float d)
{
    const uint32_t u = __float_as_uint(d);
    return u ^ ((u >> 31) ? 0xffffffffu : 0x80000000u);
}

__device__ __forceinline__ float unkey_signed(uint32_t k)
{
    return __uint_as_float(k ^ ((k >> 31) ? 0x80000000u : 0xffffffffu));
}

// One count per valid lane into h[bin].  (Adding the lanes of a warp that
// share a bin first, through match.any, was measured slower: 1844 against
// 1257 us per call at 2^27 tokens.)
__device__ __forceinline__ void hist_add(uint32_t *h, uint32_t bin, bool valid)
{
    if (valid)
        atomicAdd(h + bin, 1u);
}

template <int PASS>
struct PassShape;
template <>
struct PassShape<1> {
    static constexpr int NH = 1, NB = MON_BINS1, SHIFT = 21, KEEP = 32;   // KEEP: prefix bits compared
};
template <>
struct PassShape<2> {
    static constexpr int NH = MON_TARGETS, NB = MON_BINS2, SHIFT = 10, KEEP = 11;
};
template <>
struct PassShape<3> {
    static constexpr int NH = MON_TARGETS, NB = MON_BINS3, SHIFT = 0, KEEP = 22;
};

template <int PASS>
constexpr int pass_smem_bytes() { return PassShape<PASS>::NH * PassShape<PASS>::NB * 4; }

// One token of pass PASS (all lanes call it; `valid` false past the end).
template <int PASS>
__device__ __forceinline__ void pass_token(uint32_t *sh, const uint32_t (&pref)[MON_TARGETS], float d, bool m,
                                           bool valid,
                                           float tau, int &n_used, int &n_ext)
{
    using P = PassShape<PASS>;
    const bool used = valid && m && fabsf(d) <= FLT_MAX;
    const uint32_t ka = key_abs(d), kd = key_signed(d);
    if (PASS == 1) {   // the |delta| histogram follows from delta's (see mon_select_kernel<1>)
        hist_add(sh, kd >> P::SHIFT, used);
        n_used += static_cast<int>(used);
        n_ext += static_cast<int>(used && fabsf(d) > tau);
    } else {
#pragma unroll
        for (int j = 0; j < MON_TARGETS; ++j) {
            const uint32_t k = j < 2 ? ka : kd;
            const bool in = used && (k >> (32 - P::KEEP)) == (pref[j] >> (32 - P::KEEP));
            if (__any_sync(0xffffffffu, in))
                hist_add(sh + j * P::NB, (k >> P::SHIFT) & (P::NB - 1), in);
        }
    }
}

template <int PASS>
__global__ void __launch_bounds__(MON_THREADS, MON_CTAS_PER_SM) mon_pass_kernel(const MonArgs a)
{
    using P = PassShape<PASS>;
    extern __shared__ __align__(16) uint32_t mon_sh[];
    __shared__ uint32_t pref[MON_TARGETS];
    __shared__ int empty_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < P::NH * P::NB; i += MON_THREADS)
        mon_sh[i] = 0u;
    pdl_wait();   // the state comes from the previous kernel (or the memset)
    pdl_launch_dependents();
    if (tid < MON_TARGETS)
        pref[tid] = a.st->prefix[tid];
    if (tid == 0)
        empty_s = a.st->empty;
    __syncthreads();
    if (PASS > 1 && empty_s)   // uniform over the CTA
        return;
    uint32_t pr[MON_TARGETS];   // in registers: the histogram atomics may alias shared memory
#pragma unroll
    for (int j = 0; j < MON_TARGETS; ++j)
        pr[j] = pref[j];
    const int64_t N = a.N;
    const int64_t G = (N + 3) >> 2;   // 4-token groups; groups below `full` have 4 tokens
    const int64_t full = N >> 2;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * MON_THREADS;
    int n_used = 0, n_ext = 0;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * MON_THREADS + warp * 32; base < G;
         base += stride * MON_UNROLL) {   // uniform over the warp
        float4 lt[MON_UNROLL], lr[MON_UNROLL];
        uint32_t mk[MON_UNROLL];
#pragma unroll
        for (int u = 0; u < MON_UNROLL; ++u) {
            const int64_t g = base + lane + u * stride;
            if (g < full) {
                lt[u] = __ldcs(reinterpret_cast<const float4 *>(a.l_tr) + g);
                lr[u] = __ldcs(reinterpret_cast<const float4 *>(a.l_ro) + g);
                mk[u] = __ldcs(reinterpret_cast<const unsigned int *>(a.mask) + g);
            } else {
                float v[4] = {0.f, 0.f, 0.f, 0.f}, w[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t mm = 0u;
                for (int i = 0; i < 4 && g < G && 4 * g + i < N; ++i) {   // the ragged last group
                    v[i] = a.l_tr[4 * g + i];
                    w[i] = a.l_ro[4 * g + i];
                    mm |= static_cast<uint32_t>(a.mask[4 * g + i] != 0) << (8 * i);
                }
                lt[u] = make_float4(v[0], v[1], v[2], v[3]);
                lr[u] = make_float4(w[0], w[1], w[2], w[3]);
                mk[u] = mm;
            }
        }
#pragma unroll
        for (int u = 0; u < MON_UNROLL; ++u) {
            const int64_t g = base + lane + u * stride;
            const float d[4] = {__fsub_rn(lt[u].x, lr[u].x), __fsub_rn(lt[u].y, lr[u].y),
                                __fsub_rn(lt[u].z, lr[u].z), __fsub_rn(lt[u].w, lr[u].w)};
            uint32_t flags = 0u;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const bool valid = g < G && 4 * g + i < N;
                const bool m = ((mk[u] >> (8 * i)) & 0xffu) != 0u;
                const int before = n_ext;
                pass_token<PASS>(mon_sh, pr, d[i], m, valid, a.tau_tok, n_used, n_ext);
                flags |= static_cast<uint32_t>(n_ext != before) << (8 * i);
            }
            if (PASS == 1 && a.reject) {
                if (g < full)
                    __stcs(reinterpret_cast<unsigned int *>(a.reject) + g, flags);
                else
                    for (int i = 0; i < 4 && g < G && 4 * g + i < N; ++i)
                        a.reject[4 * g + i] = static_cast<uint8_t>((flags >> (8 * i)) & 1u);
            }
        }
    }
    if (PASS == 1) {
        const int wu = __reduce_add_sync(0xffffffffu, n_used);
        const int we = __reduce_add_sync(0xffffffffu, n_ext);
        if (lane == 0) {
            atomicAdd(&a.st->n_used, static_cast<unsigned long long>(wu));
            atomicAdd(&a.st->n_extreme, static_cast<unsigned long long>(we));
        }
    }
    __syncthreads();
    uint32_t *gh = PASS == 1 ? a.hist1 : PASS == 2 ? a.hist2 : a.hist3;
    for (int i = tid; i < P::NH * P::NB; i += MON_THREADS) {
        const uint32_t c = mon_sh[i];
        if (c != 0u)
            atomicAdd(gh + i, c);
    }
}

// Per target (warp j): the bin of the current pass that holds the target's
// rank, and the rank left inside it.  PASS 1 first turns n_used into ranks;
// PASS 3 then writes the record.  One CTA of MON_TARGETS warps.
template <int PASS>
__global__ void __launch_bounds__(MON_TARGETS * 32) mon_select_kernel(const MonArgs a)
{
    using P = PassShape<PASS>;
    const int tid = threadIdx.x, lane = tid & 31, j = tid >> 5;
    MonState *st = a.st;
    pdl_wait();   // the histograms come from mon_pass_kernel<PASS>
    pdl_launch_dependents();
    if (PASS == 1) {
        if (tid == 0) {
            const long long n = static_cast<long long>(st->n_used);
            st->empty = n == 0;
            for (int i = 0; i < MON_TARGETS / 2 && n > 0; ++i) {
                const double h = static_cast<double>(n - 1) * level(i);
                const double fl = floor(h);
                const long long k = static_cast<long long>(fl);
                st->rank[2 * i] = k;
                st->rank[2 * i + 1] = k + 1 < n ? k + 1 : k;
                st->frac[i] = h - fl;
            }
        }
        __syncthreads();
    }
    if (!st->empty) {
        // Pass 1 counted delta's key only.  |delta| has a clear top bit, and
        // its bin b holds the positive deltas of delta-bin 1024 + b and the
        // negative ones of delta-bin 1023 - b (the sign-flipped key).
        const bool abs1 = PASS == 1 && j < 2;
        const uint32_t *h = PASS == 1 ? a.hist1 : PASS == 2 ? a.hist2 + j * P::NB : a.hist3 + j * P::NB;
        auto count = [&](int b) -> long long {
            return abs1 ? static_cast<long long>(h[1024 + b]) + h[1023 - b] : static_cast<long long>(h[b]);
        };
        const long long r = st->rank[j];
        const int SEG = (abs1 ? 1024 : P::NB) / 32;   // bins per lane
        long long c = 0;
        for (int b = 0; b < SEG; ++b)
            c += count(lane * SEG + b);
        long long incl = c;   // inclusive prefix over lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += v;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, incl > r);
        int bin = -1;
        long long before = 0;
        if (hit != 0u) {
            const int L = __ffs(hit) - 1;
            if (lane == L) {
                long long cum = incl - c;
                for (int b = 0; b < SEG; ++b) {
                    const long long hb = count(lane * SEG + b);
                    if (cum + hb > r) {
                        bin = lane * SEG + b;
                        before = cum;
                        break;
                    }
                    cum += hb;
                }
            }
            bin = __shfl_sync(0xffffffffu, bin, L);
            before = __shfl_sync(0xffffffffu, before, L);
        }
        if (lane == 0) {
            if (bin < 0) {   // cannot happen when the counts are consistent
                atomicCAS(a.status, 0, static_cast<int>(TIM_ERR_BAD_INPUT));
                st->empty = 1;
            } else {
                st->rank[j] = r - before;
                st->prefix[j] |= static_cast<uint32_t>(bin) << P::SHIFT;
            }
        }
    }
    if (PASS != 3)
        return;
    __syncthreads();
    if (tid != 0)
        return;
    const unsigned long long n = st->n_used, ne = st->n_extreme;
    double *o = a.out;
    o[TIM_MON_N_USED] = static_cast<double>(n);
    o[TIM_MON_N_EXTREME] = static_cast<double>(ne);
    o[TIM_MON_FRAC_EXTREME] = n > 0 ? static_cast<double>(ne) / static_cast<double>(n) : 0.0;
    if (st->empty) {
        const double nan = __longlong_as_double(0x7ff8000000000000ll);
        o[TIM_MON_P95_ABS_DELTA] = o[TIM_MON_RATIO_Q01] = o[TIM_MON_RATIO_Q50] = o[TIM_MON_RATIO_Q99] = nan;
        return;
    }
    const double a0 = __uint_as_float(st->prefix[0]), a1 = __uint_as_float(st->prefix[1]);
    o[TIM_MON_P95_ABS_DELTA] = a0 + st->frac[0] * (a1 - a0);
    const int field[3] = {TIM_MON_RATIO_Q01, TIM_MON_RATIO_Q50, TIM_MON_RATIO_Q99};
    for (int i = 1; i < MON_TARGETS / 2; ++i) {
        const double r0 = expf(unkey_signed(st->prefix[2 * i]));
        const double r1 = expf(unkey_signed(st->prefix[2 * i + 1]));
        o[field[i - 1]] = r0 + st->frac[i] * (r1 - r0);
    }
}

template <typename K>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, const MonArgs &a)
{
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

} // namespace

cudaError_t monitor_prepare_device()
{
    cudaError_t e = cudaFuncSetAttribute(mon_pass_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         pass_smem_bytes<1>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mon_pass_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 pass_smem_bytes<2>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mon_pass_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 pass_smem_bytes<3>());
    return e;
}

cudaError_t monitor_launch(const MonArgs &a, int num_sms, cudaStream_t stream)
{
    cudaError_t e = cudaMemsetAsync(a.st, 0, MON_WORKSPACE_BYTES, stream);
    if (e != cudaSuccess)
        return e;
    const int64_t groups = (a.N + 3) / 4;
    const int64_t want = (groups + MON_THREADS - 1) / MON_THREADS;
    const dim3 grid(static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(want, static_cast<int64_t>(MON_CTAS_PER_SM) * num_sms))));
    const dim3 block(MON_THREADS), sel(MON_TARGETS * 32);
    if ((e = launch_pdl(mon_pass_kernel<1>, grid, block, pass_smem_bytes<1>(), stream, a)) != cudaSuccess ||
        (e = launch_pdl(mon_select_kernel<1>, dim3(1), sel, 0, stream, a)) != cudaSuccess ||
        (e = launch_pdl(mon_pass_kernel<2>, grid, block, pass_smem_bytes<2>(), stream, a)) != cudaSuccess ||
        (e = launch_pdl(mon_select_kernel<2>, dim3(1), sel, 0, stream, a)) != cudaSuccess ||
        (e = launch_pdl(mon_pass_kernel<3>, grid, block, pass_smem_bytes<3>(), stream, a)) != cudaSuccess)
        return e;
    return launch_pdl(mon_select_kernel<3>, dim3(1), sel, 0, stream, a);
}

} // namespace tim
