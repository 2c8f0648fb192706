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
// The eight order statistics (two per quantile) are found exactly, on 32-bit
// keys that order like the values (|delta|: its bits; delta: sign-flipped
// bits).  Counts are integers, so thread order cannot change them: the
// selected tokens are exactly the ones a sort would pick.
//   mon_sample_kernel   a histogram (14 key bits) of up to 1024 evenly spaced
//                       runs of 1024 consecutive tokens; its last CTA sets,
//                       per quantile, key bounds [lo, hi] around the sample's
//                       quantile, six standard deviations of its rank wide;
//   mon_scan_kernel     the one full pass (bulk-copied chunks): n_used,
//                       n_extreme, rejection flags and, per quantile, the used
//                       tokens below lo and the keys inside [lo, hi]
//                       (typically a few percent), kept in a list with the
//                       histogram of their offsets' high digit (top 16 bits of
//                       key - lo); its last CTA takes the ranks from n_used,
//                       checks that each quantile's order statistics fall
//                       inside its list (else, or if a list overflowed, the
//                       selection runs over all tokens) and finds each
//                       target's high digit;
//   mon_select_kernel   one pass over the lists keeps, per target, the low
//                       digits of the keys in its high bin (as values, or as a
//                       histogram when there are many); the last CTA selects
//                       the low digit and writes the record.  Over all tokens
//                       instead it runs a radix selection in three digit
//                       passes (11, 11, 10 bits) with grid barriers between
//                       them (a cooperative launch).
// The bounds only decide how much work the selection does; the result is the
// same either way.
#include <algorithm>
#include <cfloat>
#include <cmath>
#include <type_traits>

#include "monitor_internal.h"
#include "tim_internal.h"
#include "tim_ptx.cuh"
#include "../../include/tim.h"

namespace tim {
namespace {

constexpr int SAMPLE_SHIFT = 18;                         // sample bins: key >> 18
constexpr int SBD = 1 << (32 - SAMPLE_SHIFT);            // 16384 bins of delta's key
constexpr int SBA = 1 << (31 - SAMPLE_SHIFT);            // 8192 of |delta|'s key
static_assert(SBD == MON_SBINS, "sample histogram room");
constexpr double kSigmas = 6.0;                          // width of the bounds in rank standard deviations

// Quantile levels: |delta| at 0.95 (quantile 0), the ratio at 0.01, 0.5, 0.99.
__device__ __forceinline__ double level(int i)
{
    return i == 0 ? 0.95 : i == 1 ? 0.01 : i == 2 ? 0.5 : 0.99;
}

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

__device__ __forceinline__ bool usable(bool m, float d) { return m && fabsf(d) <= FLT_MAX; }

// delta = l_train - l_rollout with a zero always +0: -0 and +0 are the same
// value (and e^-0 = e^+0), so every kernel below sees one key for zero, and a
// bound between the two zeros' keys never splits equal values.
__device__ __forceinline__ float delta_of(float lt, float lr) { return __fadd_rn(__fsub_rn(lt, lr), 0.0f); }

// Tokens of a grid-stride pass in 4-token groups g (16-byte loads; the ragged
// last group by plain loads).  Calls f(g, d[4], m[4], valid[4]) on every lane
// of the warp, UNROLL groups loaded before the first use.
template <int UNROLL, typename F>
__device__ __forceinline__ void for_token_groups(const MonArgs &a, F &&f)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t N = a.N;
    const int64_t G = (N + 3) >> 2;
    const int64_t full = N >> 2;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * MON_THREADS;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * MON_THREADS + warp * 32; base < G;
         base += stride * UNROLL) {   // uniform over the warp
        float4 lt[UNROLL], lr[UNROLL];
        uint32_t mk[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t g = base + lane + u * stride;
            if (g < full) {
                lt[u] = __ldcs(reinterpret_cast<const float4 *>(a.l_tr) + g);
                lr[u] = __ldcs(reinterpret_cast<const float4 *>(a.l_ro) + g);
                mk[u] = __ldcs(reinterpret_cast<const unsigned int *>(a.mask) + g);
            } else {
                float v[4] = {0.f, 0.f, 0.f, 0.f}, w[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t mm = 0u;
                for (int i = 0; i < 4 && g < G && 4 * g + i < N; ++i) {
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
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t g = base + lane + u * stride;
            const float d[4] = {delta_of(lt[u].x, lr[u].x), delta_of(lt[u].y, lr[u].y),
                                delta_of(lt[u].z, lr[u].z), delta_of(lt[u].w, lr[u].w)};
            bool m[4], valid[4];
            const bool whole = g < full;   // all four tokens exist
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                valid[i] = whole || (g < G && 4 * g + i < N);
                m[i] = ((mk[u] >> (8 * i)) & 0xffu) != 0u;
            }
            f(g, d, m, valid);
        }
    }
}

// ---------------------------------------------------------------- histogram search
// Histogram segments in registers, loaded 16 bytes at a time (all in flight
// at once) from global memory written by atomics (read through L2).
template <int SEG>
__device__ __forceinline__ void load_segment(const uint32_t *p, uint32_t (&v)[SEG])   // p 16-byte aligned
{
#pragma unroll
    for (int i = 0; i < SEG / 4; ++i) {
        const uint4 x = __ldcg(reinterpret_cast<const uint4 *>(p) + i);
        v[4 * i] = x.x;
        v[4 * i + 1] = x.y;
        v[4 * i + 2] = x.z;
        v[4 * i + 3] = x.w;
    }
}

// |delta|'s bins [c0, c0 + SEG) from delta's histogram h of 2 half bins: a
// clear top bit means |delta|'s bin c holds the positive deltas of delta's bin
// half + c and the negative ones of bin half - 1 - c.
template <int SEG>
__device__ __forceinline__ void load_abs_segment(const uint32_t *h, int half, int c0, uint32_t (&v)[SEG])
{
    uint32_t pos[SEG], neg[SEG];
    load_segment<SEG>(h + half + c0, pos);
    load_segment<SEG>(h + half - c0 - SEG, neg);   // neg[SEG - 1 - x] = bin half - 1 - (c0 + x)
#pragma unroll
    for (int x = 0; x < SEG; ++x)
        v[x] = pos[x] + neg[SEG - 1 - x];
}

// Counts here stay below 2^31 (N < 2^31 tokens, a sample of 2^20), so 32-bit
// sums and ranks are exact.
template <int SEG>
__device__ __forceinline__ uint32_t segment_total(const uint32_t (&v)[SEG])
{
    static_assert(SEG % 8 == 0, "eight partial sums");
    uint32_t p[8];   // eight independent chains: a short dependency depth
#pragma unroll
    for (int t = 0; t < 8; ++t)
        p[t] = v[t];
#pragma unroll
    for (int x = 8; x < SEG; ++x)
        p[x % 8] += v[x];
    return ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
}

// ---------------------------------------------------------------- sample and bounds
// For quantile q at level L with m sampled used tokens: sample ranks
// floor(L (m - 1)) - w and ceil(L (m - 1)) + w, w = six standard deviations of
// a sample quantile's rank (sqrt(m L (1 - L))) + 2; lo = the lowest key of the
// bin holding the first (0 when that rank is at or below the sample's first),
// hi = the highest key of the bin holding the second (all ones when at or
// above the sample's last).  The ranks are a heuristic (a rank off by one only
// moves a bound; the check after the full pass keeps the result exact), so
// they are taken in fp32.  Run by one CTA of MON_THREADS threads on the
// global sample histogram of delta's key, seen as 512 rows of 32 bins: warp w
// loads rows [64 w, 64 w + 64), lane l bin l of each (coalesced, all in
// flight at once), copies them to shared memory `H` (SBD words) and sums each
// row (one warp reduction per row).  |delta|'s row k (its bins 32 k .. 32 k +
// 31, bin c holding delta's bins SBA - 1 - c and SBA + c) is delta's rows
// SBA / 32 + k and SBA / 32 - 1 - k, so its total is theirs.  Warps 0 and 1
// take the prefix sums of the 512 delta and 256 |delta| row totals; then warp
// b finds bound b's bin: the first row whose prefix exceeds the rank R (two
// ballots), then, in that row, the first bin whose cumulative count exceeds
// R (a warp scan and a ballot).
__device__ void compute_bounds(const MonArgs &a, uint32_t *H)
{
    constexpr int ROWS = SBD / 32, AROWS = SBA / 32;   // 512 and 256
    __shared__ uint32_t rowt[ROWS];                    // delta's row totals
    __shared__ uint32_t rowp[ROWS], arowp[AROWS];      // inclusive prefix sums of delta's and |delta|'s
    __shared__ long long R_s[2 * MON_QUANTILES];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    MonState *st = a.st;
    static_assert(ROWS == 64 * (MON_THREADS / 32) && AROWS == 32 * 8 && ROWS == 32 * 16 &&
                      MON_THREADS / 32 == 2 * MON_QUANTILES, "row split; a warp per bound");
    uint32_t v[64];
    const uint32_t *row0 = a.shist + warp * 2048 + lane;
#pragma unroll
    for (int r = 0; r < 64; ++r)
        v[r] = __ldcg(row0 + 32 * r);
    const long long m = static_cast<long long>(__ldcg(&st->sample_used));
    if (tid < 2 * MON_QUANTILES) {
        const float L = static_cast<float>(level(tid >> 1));
        const float j = static_cast<float>(m - 1) * L;
        const long long w = static_cast<long long>(ceilf(static_cast<float>(kSigmas) *
                                                         sqrtf(static_cast<float>(m) * L * (1.f - L)))) + 2;
        R_s[tid] = (tid & 1) == 0 ? static_cast<long long>(floorf(j)) - w : static_cast<long long>(ceilf(j)) + w;
    }
    uint32_t t0 = 0, t1 = 0;   // lane l: the totals of the warp's rows l and 32 + l
#pragma unroll
    for (int r = 0; r < 64; ++r) {
        H[warp * 2048 + 32 * r + lane] = v[r];
        const uint32_t t = __reduce_add_sync(0xffffffffu, v[r]);
        if (lane == (r & 31)) {
            if (r < 32)
                t0 = t;
            else
                t1 = t;
        }
    }
    rowt[warp * 64 + lane] = t0;
    rowt[warp * 64 + 32 + lane] = t1;
    __syncthreads();
    if (warp == 0) {   // delta's rows: lane l the rows [16 l, 16 l + 16)
        uint32_t x[16], run = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            run += rowt[16 * lane + i];
            x[i] = run;
        }
        uint32_t incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += y;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
            rowp[16 * lane + i] = incl - run + x[i];
    } else if (warp == 1) {   // |delta|'s rows: lane l the rows [8 l, 8 l + 8)
        uint32_t x[8], run = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int k = 8 * lane + i;
            run += rowt[AROWS + k] + rowt[AROWS - 1 - k];
            x[i] = run;
        }
        uint32_t incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += y;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
            arowp[8 * lane + i] = incl - run + x[i];
    }
    __syncthreads();
    // warp b: bound b (quantile b / 2; b even: lo, odd: hi)
    const int b = warp, q = b >> 1;
    const long long R = R_s[b];
    int bin = -1;
    if (m > 0 && R > 0 && R < m - 1) {   // then some bin holds R: the last prefix is m
        const uint32_t r = static_cast<uint32_t>(R);
        const uint32_t *pp = q == 0 ? arowp : rowp;
        const int per = q == 0 ? AROWS / 32 : ROWS / 32;   // rows per lane in the first ballot
        const unsigned big = __ballot_sync(0xffffffffu, pp[per * lane + per - 1] > r);
        const int L = __ffs(big) - 1;                       // big != 0: the last prefix is m > r
        const unsigned in = __ballot_sync(0xffffffffu, lane < per && pp[per * L + lane] > r);
        const int row = per * L + __ffs(in) - 1;
        const uint32_t before = row > 0 ? pp[row - 1] : 0u;
        uint32_t c = q == 0 ? H[SBA + 32 * row + lane] + H[SBA - 1 - 32 * row - lane] : H[32 * row + lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, c, o);
            if (lane >= o)
                c += y;
        }
        bin = 32 * row + __ffs(__ballot_sync(0xffffffffu, before + c > r)) - 1;
    }
    if (lane == 0) {
        if ((b & 1) == 0)
            st->lo[q] = bin < 0 ? 0u : static_cast<uint32_t>(bin) << SAMPLE_SHIFT;
        else
            st->hi[q] = bin < 0 ? 0xffffffffu
                                : (static_cast<uint32_t>(bin) << SAMPLE_SHIFT) | ((1u << SAMPLE_SHIFT) - 1u);
    }
}

// Adds the non-zero words of a shared-memory histogram of `words` bins to
// the global one (16-byte shared-memory reads, all threads of the CTA).
template <int WORDS>
__device__ __forceinline__ void flush_histogram(const uint32_t *sh, uint32_t *gh)
{
    static_assert(WORDS % (4 * MON_THREADS) == 0, "whole 16-byte reads per thread");
#pragma unroll
    for (int k = 0; k < WORDS / (4 * MON_THREADS); ++k) {
        const int i = threadIdx.x + k * MON_THREADS;
        const uint4 x = reinterpret_cast<const uint4 *>(sh)[i];
        if (x.x != 0u)
            atomicAdd(gh + 4 * i, x.x);
        if (x.y != 0u)
            atomicAdd(gh + 4 * i + 1, x.y);
        if (x.z != 0u)
            atomicAdd(gh + 4 * i + 2, x.z);
        if (x.w != 0u)
            atomicAdd(gh + 4 * i + 3, x.w);
    }
}

template <int WORDS>
__device__ __forceinline__ void zero_histogram(uint32_t *sh)
{
    static_assert(WORDS % (4 * MON_THREADS) == 0, "whole 16-byte writes per thread");
#pragma unroll
    for (int k = 0; k < WORDS / (4 * MON_THREADS); ++k)
        reinterpret_cast<uint4 *>(sh)[threadIdx.x + k * MON_THREADS] = make_uint4(0u, 0u, 0u, 0u);
}

// Is this CTA the last of the grid to get here?  Every thread's global writes
// before the call are ordered before the ticket (a fence per thread, then the
// barrier); the last CTA fences again before it reads what the others wrote.
__device__ __forceinline__ bool last_cta(unsigned *ticket)
{
    __shared__ int last_s;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        last_s = atomicAdd(ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!last_s)
        return false;
    __threadfence();
    return true;
}

// Run r: MON_SAMPLE_RUN tokens from s = g (N - R) / 63 rounded down to a
// multiple of 4, plus j R / 16 (g = r / 16, j = r mod 16, R = kSampleRegion;
// runs back to back when they cover the batch); CTA c takes runs c, c +
// gridDim, ..., kRunsAtOnce of them loaded before any is used, into a
// shared-memory histogram of delta's key (|delta|'s follows from it), thread
// i the tokens s + 4i .. s + 4i + 3 (one 16-byte load per array), and adds
// the non-zero bins to the global histogram.  The CTA that finishes last
// computes the bounds.
constexpr int kRunsAtOnce = 8;   // with one CTA per SM, all 1024 runs in one round of loads
constexpr int64_t kSampleRegion = int64_t(1) << 18;   // tokens of one of the sample's 64 regions
static_assert(MON_SAMPLE_RUNS == 64 * 16 && kSampleRegion / 16 >= MON_SAMPLE_RUN &&
                  kSampleRegion <= int64_t(MON_SAMPLE_RUNS) * MON_SAMPLE_RUN,
              "64 regions of 16 runs, within the batch whenever the sample does not cover it");
static_assert(MON_SAMPLE_RUN == 4 * MON_THREADS, "a run is one 4-token group per thread");
__global__ void __launch_bounds__(MON_THREADS) mon_sample_kernel(const MonArgs a)
{
    extern __shared__ __align__(16) uint32_t sh[];   // [SBD] delta's key
    const int tid = threadIdx.x, lane = tid & 31;
    zero_histogram<SBD>(sh);
    __syncthreads();
    pdl_wait();
    {   // the fine histograms of the full pass and the selection pass start at zero
        constexpr size_t n4 = (MON_HIF_WORDS + MON_LOF_WORDS) / 4;
        static_assert((MON_HIF_WORDS + MON_LOF_WORDS) % 4 == 0, "whole 16-byte stores");
        uint4 *z = reinterpret_cast<uint4 *>(a.hif);   // hif and lof are adjacent
        for (size_t i = static_cast<size_t>(blockIdx.x) * MON_THREADS + tid; i < n4;
             i += static_cast<size_t>(gridDim.x) * MON_THREADS)
            z[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    const int64_t N = a.N;
    const int64_t cover = static_cast<int64_t>(MON_SAMPLE_RUNS) * MON_SAMPLE_RUN;
    const int64_t runs = std::min<int64_t>(MON_SAMPLE_RUNS, (N + MON_SAMPLE_RUN - 1) / MON_SAMPLE_RUN);
    int used = 0;
    for (int64_t r0 = blockIdx.x; r0 < runs; r0 += kRunsAtOnce * gridDim.x) {
        float v[kRunsAtOnce][4], w[kRunsAtOnce][4];
        uint32_t mm[kRunsAtOnce];
#pragma unroll
        for (int k = 0; k < kRunsAtOnce; ++k) {
            const int64_t r = r0 + k * static_cast<int64_t>(gridDim.x);
            mm[k] = 0u;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                v[k][i] = w[k][i] = 0.f;
            if (r >= runs)
                continue;
            // 64 regions of kSampleRegion tokens spread over the batch, 16 runs
            // spread over each region: the runs still come from 1024 places
            // (sequences) but touch ~1/3 of the pages that runs spread over the
            // whole batch touch (the sample's loads wait mostly on page-table
            // walks)
            const int64_t s0 =
                N <= cover ? r * MON_SAMPLE_RUN
                           : (((r >> 4) * (N - kSampleRegion) / 63) & ~int64_t(3)) + (r & 15) * (kSampleRegion / 16);
            const int64_t s1 = std::min<int64_t>(N, s0 + MON_SAMPLE_RUN);
            const int64_t t = s0 + 4 * tid;
            if (t + 4 <= s1) {
                const float4 x = __ldcs(reinterpret_cast<const float4 *>(a.l_tr + t));
                const float4 y = __ldcs(reinterpret_cast<const float4 *>(a.l_ro + t));
                mm[k] = __ldcs(reinterpret_cast<const unsigned int *>(a.mask + t));
                v[k][0] = x.x, v[k][1] = x.y, v[k][2] = x.z, v[k][3] = x.w;
                w[k][0] = y.x, w[k][1] = y.y, w[k][2] = y.z, w[k][3] = y.w;
            } else {
                for (int i = 0; i < 4 && t + i < s1; ++i) {
                    v[k][i] = a.l_tr[t + i];
                    w[k][i] = a.l_ro[t + i];
                    mm[k] |= static_cast<uint32_t>(a.mask[t + i] != 0) << (8 * i);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kRunsAtOnce; ++k)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float d = delta_of(v[k][i], w[k][i]);
                if (usable(((mm[k] >> (8 * i)) & 0xffu) != 0u, d)) {
                    atomicAdd(sh + (key_signed(d) >> SAMPLE_SHIFT), 1u);
                    ++used;
                }
            }
    }
    used = __reduce_add_sync(0xffffffffu, used);
    if (lane == 0 && used)
        atomicAdd(&a.st->sample_used, static_cast<unsigned long long>(used));
    __syncthreads();
    // The full pass's CTAs may launch now (they wait for the bounds).  (Earlier,
    // when this kernel ran two CTAs per SM, they took the room of its second
    // CTA, which then started ~10 us late.)
    pdl_launch_dependents();
    flush_histogram<SBD>(sh, a.shist);
    if (last_cta(&a.st->ticket[0]))
        compute_bounds(a, sh);   // the CTA's histogram is spent: its room takes the global one
}

// ---------------------------------------------------------------- the full pass
// A warp takes chunks of 512 consecutive tokens (chunk w, w + warps, ...);
// its lane 0 bulk-copies them (l_train, l_rollout, mask) into a ring of
// kRing slots in shared memory, one chunk ahead of the one the warp works on;
// the ragged last chunk is read from global memory.  Lane l takes the 4-token
// groups l, l + 32, l + 64, l + 96 of the chunk.
//
// The tests run on the canonical delta itself (NaN for an unused token), with
// float thresholds equal to the key bounds: per token and quantile one compare
// for "at or above lo" (counted; the used tokens below lo are the used tokens
// less these) and one for "in [lo, hi]" (a bit in the step's mask).  The
// counts and bits are added by multiplies with `one`, so that they issue on
// the FMA pipe while the compares take the integer ALU (the ALU alone had
// bound the pass).  The keys in range are placed by a ballot when no lane has
// two of a quantile (the usual case), else by a warp scan of the counts; they
// are staged per warp and quantile in shared memory and go to the global list
// 32 at a time (one atomic reservation per 32 keys), or straight to the list
// when a step brings more than the stage holds.  (A ballot per token and
// quantile took 13% longer; a private buffer per thread 2.3x longer.)
constexpr int kScanGroups = 4;                           // 4-token groups per lane and step
constexpr int kScanTokens = 4 * kScanGroups;
constexpr int kStage = 64;                              // staged keys per warp and quantile (a step that
                                                        // does not fit writes its keys straight to the list)
constexpr int kRing = 2;                                // ring slots per warp
constexpr int kChunkTokens = 32 * kScanTokens;
constexpr int kChunkF = 4 * kChunkTokens;               // bytes of one fp32 array's chunk
constexpr int kChunkBytes = 2 * kChunkF + kChunkTokens; // l_train, l_rollout, mask
// One CTA of 16 warps per SM (rings and stages: 160 KB of shared memory).
// (Two CTAs of 8 warps per SM had the younger CTA of each SM finish ~26 us
// after the older one, ~11 % of the pass: the warp schedulers favour the
// older CTA's warps, and the pass is bound by instruction issue.)
constexpr int kScanThreads = 512;
constexpr int kScanWarps = kScanThreads / 32;
constexpr size_t kRingBytes = static_cast<size_t>(kScanWarps) * kRing * kChunkBytes;
constexpr size_t kStageBytes = sizeof(uint32_t) * kScanWarps * MON_QUANTILES * kStage;
constexpr size_t kScanSmem = kRingBytes + kStageBytes + 8 * kScanWarps * kRing;
static_assert(kChunkF % 16 == 0 && kChunkBytes % 16 == 0 && kRingBytes % 16 == 0, "bulk copies stay 16-byte aligned");

// Radix digits of a value with b significant bits (b = 32 for raw keys): pass
// 1 the top 11 (bits b-11 .. b-1), pass 2 the next 11, pass 3 the rest (<= 10).
__device__ __forceinline__ int digit_shift(int pass, int b)
{
    return pass == 1 ? max(b - 11, 0) : pass == 2 ? max(b - 22, 0) : 0;
}

template <int PASS>
__device__ __forceinline__ uint32_t digit_of(uint32_t v, int b)
{
    const int s = digit_shift(PASS, b);
    const int top = PASS == 1 ? b : digit_shift(PASS - 1, b);
    const int width = top - s;   // <= 11
    return (v >> s) & ((1u << width) - 1u);
}

// Significant bits of hi - lo: the width of the collected keys' offsets.
__device__ __forceinline__ int span_bits_of(uint32_t lo, uint32_t hi)
{
    const uint32_t span = hi - lo;
    return span == 0u ? 0 : 32 - __clz(static_cast<int>(span));
}

// The shift that leaves the high digit (top MON_HI_BITS bits) of an offset
// key - lo of a list whose offsets have `bits` significant bits.
__device__ __forceinline__ int high_shift(int bits) { return max(bits - MON_HI_BITS, 0); }

// Collected keys of quantile q, one per lane with `has` set (a full warp
// calls): each into the list at `at` (when there is room) and into the list's
// histograms of its offset's high digit (fine: all 16 bits, in global memory;
// coarse: the top 8, in the CTA's shared-memory copy `hic_s`, added to the
// global one at the end: its few bins take most keys), lanes with the same
// digit added by one atomic (the keys near a quantile share few digits).
__device__ __forceinline__ void collect(const MonArgs &a, uint32_t *hic_s, int q, bool has, unsigned long long at,
                                        uint32_t key, uint32_t lo, int shift)
{
    uint32_t hd = has ? (key - lo) >> shift : 0xffffffffu;   // < 2^16: lo <= key <= hi
    TIM_DCHECK(!has || hd < static_cast<uint32_t>(MON_FINE), a.status, TIM_CHECK_UNIT, q, key);
    has = has && hd < static_cast<uint32_t>(MON_FINE);
    hd = has ? hd : 0xffffffffu;
    const unsigned same = __match_any_sync(0xffffffffu, hd);
    const unsigned same_c = __match_any_sync(0xffffffffu, has ? hd >> 8 : 0xffffffffu);
    if (has) {
        const int lane = threadIdx.x & 31;
        if (at < a.cap)   // kept in L2 (evict-last) for the selection pass that reads it next
            st_global_hint(a.cand + static_cast<size_t>(q) * a.cap + at, key, l2_policy_evict_last());
        if (lane == __ffs(same) - 1)
            atomicAdd(a.hif + q * MON_FINE + hd, static_cast<uint32_t>(__popc(same)));
        if (lane == __ffs(same_c) - 1)
            atomicAdd(hic_s + q * MON_COARSE + (hd >> 8), static_cast<uint32_t>(__popc(same_c)));
    }
}

__device__ __forceinline__ void flush_stage(const MonArgs &a, uint32_t *hic_s, const uint32_t *buf, int q, int n,
                                            int lane, uint32_t lo, int shift)
{
    unsigned long long base = 0;
    if (lane == 0)
        base = atomicAdd(a.hot + q * MON_HOT_STRIDE, static_cast<unsigned long long>(n));
    base = __shfl_sync(0xffffffffu, base, 0);
    collect(a, hic_s, q, lane < n, base + lane, lane < n ? buf[lane] : 0u, lo, shift);
}

// Float thresholds equal to the key bounds on canonical finite deltas:
// key(delta) >= lo  <=>  delta >= lo_threshold(lo), key(delta) <= hi  <=>
// delta <= hi_threshold(hi) (-inf / +inf where every or no finite delta
// qualifies).  Keys of finite canonical deltas: [key(-FLT_MAX), key(-min
// subnormal)] and [key(+0), key(FLT_MAX)].
constexpr uint32_t kKeyNegMax = 0x00800000u;   // key(-FLT_MAX)
constexpr uint32_t kKeyNegMin = 0x7ffffffeu;   // key(-smallest subnormal)
constexpr uint32_t kKeyZero = 0x80000000u;     // key(+0)
constexpr uint32_t kKeyPosMax = 0xff7fffffu;   // key(FLT_MAX)

__device__ __forceinline__ float signed_lo_threshold(uint32_t lo)
{
    if (lo <= kKeyNegMax)
        return -INFINITY;
    if (lo > kKeyPosMax)
        return INFINITY;
    if (lo > kKeyNegMin && lo <= kKeyZero)
        return 0.0f;
    return unkey_signed(lo);
}

__device__ __forceinline__ float signed_hi_threshold(uint32_t hi)
{
    if (hi >= kKeyPosMax)
        return INFINITY;
    if (hi < kKeyNegMax)
        return -INFINITY;
    if (hi >= kKeyNegMin && hi < kKeyZero)
        return unkey_signed(kKeyNegMin);
    return unkey_signed(hi);
}

__device__ __forceinline__ float abs_lo_threshold(uint32_t lo)
{
    return lo > 0x7f7fffffu ? INFINITY : __uint_as_float(lo);
}

__device__ __forceinline__ float abs_hi_threshold(uint32_t hi)
{
    return hi >= 0x7f7fffffu ? INFINITY : __uint_as_float(hi);
}

// Per token: the used test (mask byte and finite delta), the count of used
// tokens and the rejection flag, both added with a multiply by `one` (= 1, read
// from memory) so that they issue on the FMA pipe, not the integer ALU; the
// delta itself, NaN for an unused token (it then passes no test below).
__device__ __forceinline__ float token_delta(float d, uint32_t mk, uint32_t byte_sel, float tau, uint32_t one,
                                             uint32_t flag_bit, int &n_used, uint32_t &flags)
{
    float v;
    asm("{\n\t.reg .pred pm, pu, pe;\n\t.reg .u32 b;\n\t.reg .f32 fa;\n\t"
        "and.b32 b, %4, %5;\n\t"
        "setp.ne.u32 pm, b, 0;\n\t"
        "abs.f32 fa, %3;\n\t"
        "setp.le.and.f32 pu, fa, 0f7F7FFFFF, pm;\n\t"
        "@pu mad.lo.u32 %0, %7, %7, %0;\n\t"
        "setp.gt.and.f32 pe, fa, %6, pu;\n\t"
        "@pe mad.lo.u32 %1, %7, %8, %1;\n\t"
        "selp.f32 %2, %3, 0f7FFFFFFF, pu;\n\t}"
        : "+r"(n_used), "+r"(flags), "=f"(v)
        : "f"(d), "r"(mk), "r"(byte_sel), "f"(tau), "r"(one), "r"(flag_bit));
    return v;
}

// ge += (x >= lo); inbits += bit when lo <= x <= hi (x NaN: neither).
__device__ __forceinline__ void range_test(float x, float lo, float hi, uint32_t bit, uint32_t one, int &ge,
                                           uint32_t &inbits)
{
    asm("{\n\t.reg .pred p, r;\n\t"
        "setp.ge.f32 p, %2, %3;\n\t"
        "@p mad.lo.u32 %0, %6, %6, %0;\n\t"
        "setp.le.and.f32 r, %2, %4, p;\n\t"
        "@r mad.lo.u32 %1, %6, %5, %1;\n\t}"
        : "+r"(ge), "+r"(inbits)
        : "f"(x), "f"(lo), "f"(hi), "r"(bit), "r"(one));
}

// k[s] by a tree of selects on the bits of s.
__device__ __forceinline__ float pick(const float (&k)[kScanTokens], int s)
{
    static_assert((kScanTokens & (kScanTokens - 1)) == 0, "a power-of-two tree");
    float l[kScanTokens];
#pragma unroll
    for (int j = 0; j < kScanTokens; ++j)
        l[j] = k[j];
#pragma unroll
    for (int w = kScanTokens / 2, bit = 0; w >= 1; w >>= 1, ++bit)
#pragma unroll
        for (int j = 0; j < w; ++j)
            l[j] = ((s >> bit) & 1) ? l[2 * j + 1] : l[2 * j];
    return l[0];
}

__device__ void check_ranks(const MonArgs &a);
__device__ void select_high(const MonArgs &a);

__global__ void __launch_bounds__(kScanThreads, 1) mon_scan_kernel(const MonArgs a)
{
    extern __shared__ __align__(16) uint8_t scan_smem[];   // rings [warp][kRing], staging, barriers
    __shared__ float flo_s[MON_QUANTILES], fhi_s[MON_QUANTILES];
    __shared__ uint32_t one_s, lo_s[MON_QUANTILES];
    __shared__ int shift_s[MON_QUANTILES];
    __shared__ __align__(16) uint32_t hic_s[MON_QUANTILES * MON_COARSE];   // the lists' coarse high digits
    __shared__ int abort_s;
    volatile int *abort_flag = &abort_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned lanes_below = (1u << lane) - 1u;
    uint8_t *const ring = scan_smem + static_cast<size_t>(warp) * kRing * kChunkBytes;
    uint32_t *const stage_all = reinterpret_cast<uint32_t *>(scan_smem + kRingBytes);
    const uint32_t bar0 = smem_u32(scan_smem + kRingBytes + kStageBytes) + 8u * kRing * warp;
    if (lane == 0) {
        for (int i = 0; i < kRing; ++i)
            mbar_init(bar0 + 8u * i, 1);
        fence_mbar_init();
    }
    if (tid == 0) {
        one_s = 1u;
        abort_s = 0;
    }
    for (int i = tid; i < MON_QUANTILES * MON_COARSE; i += kScanThreads)
        hic_s[i] = 0u;
    float flo[MON_QUANTILES], fhi[MON_QUANTILES];   // set from the sample's bounds (below)
    uint32_t one = 0u;
    const int64_t N = a.N;
    const int64_t G = (N + 3) >> 2;
    const int64_t full = N >> 2;
    constexpr int64_t kChunk = 32 * kScanGroups;   // groups per warp and step: lane + 32 u
    const int64_t warps = static_cast<int64_t>(gridDim.x) * kScanWarps;
    const float tau = a.tau_tok;
    const uint64_t pol = l2_policy_evict_first();
    int n_used = 0, n_ext = 0;
    int staged[MON_QUANTILES] = {0, 0, 0, 0};   // uniform over the warp
    int at_or_above[MON_QUANTILES] = {0, 0, 0, 0};

    // Chunk c holds groups [c kChunk, (c + 1) kChunk); chunks below `whole_n`
    // are whole (bulk-copied), chunk `whole_n` is the ragged last one when N is
    // not a multiple of the chunk.  The warp takes chunks w, w + warps, ...
    // (Handing the second half out in blocks from a counter evened the warps'
    // finish times but made the pass slower: the claims' atomics on one word
    // queue up, and how much varied from one device to another.)
    const int64_t w = static_cast<int64_t>(blockIdx.x) * kScanWarps + warp;
    const int64_t whole_n = full / kChunk;
    const int64_t chunks = whole_n + (whole_n * kChunk < G ? 1 : 0);
    auto chunk_of = [&](int64_t k) -> int64_t {   // the warp's k-th chunk, -1 past the last (uniform)
        const int64_t c = w + k * warps;
        return c < chunks ? c : -1;
    };
    auto issue = [&](int slot, int64_t c) {   // lane 0: stage whole chunk c into ring slot `slot`
        if (lane != 0 || c < 0 || c >= whole_n)
            return;
        const int64_t g0 = c * kChunk;
        const uint32_t dst = smem_u32(ring + slot * kChunkBytes), bar = bar0 + 8u * slot;
        TIM_DCHECK(g0 + kChunk <= full, a.status, TIM_CHECK_UNIT, c, static_cast<uint64_t>(chunks));
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, kChunkBytes);
        bulk_load(dst, a.l_tr + 4 * g0, kChunkF, bar, pol);
        bulk_load(dst + kChunkF, a.l_ro + 4 * g0, kChunkF, bar, pol);
        bulk_load(dst + 2 * kChunkF, a.mask + 4 * g0, kChunkTokens, bar, pol);
    };

    auto step = [&](int64_t g0, const uint8_t *src, auto checked) {
        constexpr bool CHECK = decltype(checked)::value;
        const int64_t gl = g0 + lane;
        float4 lt[kScanGroups], lr[kScanGroups];
        uint32_t mk[kScanGroups];
#pragma unroll
        for (int u = 0; u < kScanGroups; ++u) {
            const int64_t g = gl + 32 * u;
            if (!CHECK) {
                lt[u] = reinterpret_cast<const float4 *>(src)[lane + 32 * u];
                lr[u] = reinterpret_cast<const float4 *>(src + kChunkF)[lane + 32 * u];
                mk[u] = reinterpret_cast<const uint32_t *>(src + 2 * kChunkF)[lane + 32 * u];
                TIM_DCHECK((mk[u] & 0xfefefefeu) == 0u, a.status, TIM_CHECK_MASK, 4 * g, mk[u]);
            } else {
                float v[4] = {0.f, 0.f, 0.f, 0.f}, x[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t mm = 0u;
                for (int i = 0; i < 4 && g < G && 4 * g + i < N; ++i) {
                    v[i] = a.l_tr[4 * g + i];
                    x[i] = a.l_ro[4 * g + i];
                    mm |= static_cast<uint32_t>(a.mask[4 * g + i] != 0) << (8 * i);
                }
                lt[u] = make_float4(v[0], v[1], v[2], v[3]);
                lr[u] = make_float4(x[0], x[1], x[2], x[3]);
                mk[u] = mm;
            }
        }
        float dv[kScanTokens];   // canonical delta, NaN when unused
        uint32_t inbits[MON_QUANTILES] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int u = 0; u < kScanGroups; ++u) {
            const int64_t g = gl + 32 * u;
            const float d[4] = {delta_of(lt[u].x, lr[u].x), delta_of(lt[u].y, lr[u].y),
                                delta_of(lt[u].z, lr[u].z), delta_of(lt[u].w, lr[u].w)};
            uint32_t flags = 0u;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int s = 4 * u + i;
                dv[s] = token_delta(d[i], mk[u], 0xffu << (8 * i), tau, one, 1u << (8 * i), n_used, flags);
                range_test(fabsf(dv[s]), flo[0], fhi[0], 1u << s, one, at_or_above[0], inbits[0]);
#pragma unroll
                for (int q = 1; q < MON_QUANTILES; ++q)
                    range_test(dv[s], flo[q], fhi[q], 1u << s, one, at_or_above[q], inbits[q]);
            }
            n_ext += __popc(flags);
            if (a.reject) {
                if (!CHECK || g < full)
                    __stcs(reinterpret_cast<unsigned int *>(a.reject) + g, flags);
                else
                    for (int i = 0; i < 4 && g < G && 4 * g + i < N; ++i)
                        a.reject[4 * g + i] = static_cast<uint8_t>((flags >> (8 * i)) & 1u);
            }
        }
#pragma unroll
        for (int q = 0; q < MON_QUANTILES; ++q) {
            const int c = __popc(inbits[q]);
            const unsigned lanes_with = __ballot_sync(0xffffffffu, c != 0);
            if (lanes_with == 0u)   // uniform over the warp
                continue;
            int excl, total;
            if (__ballot_sync(0xffffffffu, c > 1) == 0u) {
                excl = __popc(lanes_with & lanes_below);
                total = __popc(lanes_with);
            } else {
                int incl = c;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o)
                        incl += v;
                }
                total = __shfl_sync(0xffffffffu, incl, 31);
                excl = incl - c;
            }
            if (staged[q] + total > kStage) {   // rare: straight to the list, one reservation
                unsigned long long base = 0;
                if (lane == 0)
                    base = atomicAdd(a.hot + q * MON_HOT_STRIDE, static_cast<unsigned long long>(total));
                base = __shfl_sync(0xffffffffu, base, 0) + static_cast<unsigned long long>(excl);
                for (uint32_t b = inbits[q]; __any_sync(0xffffffffu, b != 0u); b &= b - 1u, ++base) {
                    const float v = b != 0u ? pick(dv, __ffs(b) - 1) : 0.f;
                    collect(a, hic_s, q, b != 0u, base, q == 0 ? key_abs(v) : key_signed(v), lo_s[q], shift_s[q]);
                }
                continue;
            }
            uint32_t *buf = stage_all + (warp * MON_QUANTILES + q) * kStage;
            int pos = staged[q] + excl;
            for (uint32_t b = inbits[q]; b != 0u; b &= b - 1u) {
                const float v = pick(dv, __ffs(b) - 1);
                buf[pos++] = q == 0 ? key_abs(v) : key_signed(v);
            }
            staged[q] += total;
            __syncwarp();
            while (staged[q] >= 32) {   // uniform over the warp
                flush_stage(a, hic_s, buf, q, 32, lane, lo_s[q], shift_s[q]);
                __syncwarp();
                for (int i = lane; i + 32 < staged[q]; i += 32) {   // move the rest down
                    const uint32_t v = buf[i + 32];
                    __syncwarp(__activemask());
                    buf[i] = v;
                }
                __syncwarp();
                staged[q] -= 32;
            }
        }
    };

    // Whole chunks through the ring; the ragged last one from global memory.
    // cs0, cs1: the chunks of ring slots 0 and 1; parity bit i: the phase of
    // slot i's next completion (a slot's barrier completes only for a staged
    // chunk).
    static_assert(kRing == 2, "two ring slots");
    int64_t cs0 = chunk_of(0);
    issue(0, cs0);
    int64_t cs1 = chunk_of(1);
    issue(1, cs1);
    // The inputs do not depend on the sample kernel (it waited for every
    // earlier write before it let this kernel start): the first two chunks are
    // in flight while the sample's last CTA sets the bounds.
    pdl_wait();
    pdl_launch_dependents();
    if (tid < MON_QUANTILES) {
        const uint32_t lo = a.st->lo[tid], hi = a.st->hi[tid];
        flo_s[tid] = tid == 0 ? abs_lo_threshold(lo) : signed_lo_threshold(lo);
        fhi_s[tid] = tid == 0 ? abs_hi_threshold(hi) : signed_hi_threshold(hi);
        lo_s[tid] = lo;
        shift_s[tid] = high_shift(span_bits_of(lo, hi));
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < MON_QUANTILES; ++q) {
        flo[q] = flo_s[q];
        fhi[q] = fhi_s[q];
    }
    one = one_s;
    uint32_t parity = 0;
    bool ok = true;
    for (int64_t k = 0;; ++k) {
        const int slot = static_cast<int>(k & 1);
        const int64_t c = slot ? cs1 : cs0;   // uniform over the warp
        if (c < 0)
            break;
        if (c < whole_n) {
            if (!mbar_wait_sleep(bar0 + 8u * slot, (parity >> slot) & 1u, abort_flag, a.wait_budget_ns)) {
                ok = false;
                break;
            }
            parity ^= 1u << slot;
            step(c * kChunk, ring + slot * kChunkBytes, std::false_type{});
        } else {
            step(c * kChunk, nullptr, std::true_type{});
        }
        __syncwarp();   // every lane has read the slot
        const int64_t cn = chunk_of(k + kRing);
        if (slot)
            cs1 = cn;
        else
            cs0 = cn;
        issue(slot, cn);
    }
    if (!ok) {   // copies may still be landing: let them, then report
        if (cs0 >= 0 && cs0 < whole_n)
            drain_wait(bar0, parity & 1u);
        if (cs1 >= 0 && cs1 < whole_n)
            drain_wait(bar0 + 8u, (parity >> 1) & 1u);
        if (lane == 0)
            atomicCAS(a.status, 0, static_cast<int>(TIM_ERR_TIMEOUT));
    }

    __syncwarp();
#pragma unroll
    for (int q = 0; q < MON_QUANTILES; ++q)
        if (staged[q] > 0)
            flush_stage(a, hic_s, stage_all + (warp * MON_QUANTILES + q) * kStage, q, staged[q], lane, lo_s[q],
                        shift_s[q]);
    // the CTA's counts (warp sums, then thread 0 adds the warps': one atomic
    // per counter and CTA)
    __shared__ int red_s[kScanWarps][2 + MON_QUANTILES];
    const int wu = __reduce_add_sync(0xffffffffu, n_used);
    const int we = __reduce_add_sync(0xffffffffu, n_ext);
    int wb[MON_QUANTILES];
#pragma unroll
    for (int q = 0; q < MON_QUANTILES; ++q)
        wb[q] = __reduce_add_sync(0xffffffffu, n_used - at_or_above[q]);
    if (lane == 0) {
        red_s[warp][0] = wu;
        red_s[warp][1] = we;
#pragma unroll
        for (int q = 0; q < MON_QUANTILES; ++q)
            red_s[warp][2 + q] = wb[q];
    }
    __syncthreads();
    for (int i = tid; i < MON_QUANTILES * MON_COARSE; i += kScanThreads)   // the CTA's coarse counts
        if (hic_s[i] != 0u)
            atomicAdd(a.hic + i, hic_s[i]);
    if (tid < 2 + MON_QUANTILES) {
        unsigned long long t = 0;
        for (int w2 = 0; w2 < kScanWarps; ++w2)
            t += static_cast<unsigned long long>(red_s[w2][tid]);
        unsigned long long *dst = tid == 0 ? &a.st->n_used : tid == 1 ? &a.st->n_extreme : &a.st->below[tid - 2];
        if (t)
            atomicAdd(dst, t);
    }
    // The last CTA: ranks and mode, then (collected lists) the targets' high digits.
    if (last_cta(&a.st->ticket[1])) {
        if (tid == 0)
            check_ranks(a);
        __syncthreads();
        if (!a.st->empty && !a.st->fallback && tid < 32 * MON_TARGETS)   // uniform over each warp
            select_high(a);
    }
}

// ---------------------------------------------------------------- ranks and mode
// Thread 0 of the full pass's last CTA.  For each quantile at level L over the
// n used tokens: h = (n - 1) L, ranks floor(h) and floor(h) + 1 (capped at
// n - 1) and the weight h - floor(h).  Each quantile's two order statistics
// must fall inside its list (below <= k, k + 1 < below + count, no overflow),
// else the selection runs over all tokens; the ranks are then taken relative
// to the list (collected) or to all tokens.
__device__ void check_ranks(const MonArgs &a)
{
    MonState *st = a.st;
    const long long n = static_cast<long long>(__ldcg(&st->n_used));
    st->empty = n == 0;
    if (n == 0)
        return;
    bool ok = true;
    long long k[MON_QUANTILES], k1[MON_QUANTILES], below[MON_QUANTILES], cnt[MON_QUANTILES];
#pragma unroll
    for (int q = 0; q < MON_QUANTILES; ++q) {   // all loads first: they are independent
        below[q] = static_cast<long long>(__ldcg(&st->below[q]));
        cnt[q] = static_cast<long long>(__ldcg(a.hot + q * MON_HOT_STRIDE));
    }
    for (int q = 0; q < MON_QUANTILES; ++q) {
        const double h = static_cast<double>(n - 1) * level(q);
        const double fl = floor(h);
        k[q] = static_cast<long long>(fl);
        k1[q] = k[q] + 1 < n ? k[q] + 1 : k[q];
        st->frac[q] = h - fl;
        ok = ok && cnt[q] <= static_cast<long long>(a.cap) && below[q] <= k[q] && k1[q] < below[q] + cnt[q];
    }
    st->fallback = ok ? 0 : 1;
    for (int q = 0; q < MON_QUANTILES; ++q) {
        const long long b = ok ? below[q] : 0;
        st->rank[2 * q] = k[q] - b;
        st->rank[2 * q + 1] = k1[q] - b;
        st->span_bits[q] = ok ? span_bits_of(st->lo[q], st->hi[q]) : 32;
    }
}


// ---------------------------------------------------------------- bin search in a warp
// The first bin x of a segment with cum + v[0] + ... + v[x] > r, or -1;
// `before` gets the count below bin x and `in` its count.
template <int SEG>
__device__ __forceinline__ int find_bin_in_segment(const uint32_t (&v)[SEG], uint32_t cum, uint32_t r,
                                                   uint32_t &before, uint32_t &in)
{
    int bin = -1;
#pragma unroll
    for (int x = 0; x < SEG; ++x) {
        if (bin < 0 && cum + v[x] > r) {
            bin = x;
            before = cum;
            in = v[x];
        }
        cum += v[x];
    }
    return bin;
}

// The bin of a histogram that holds rank r, lane l holding bins [l SEG,
// (l + 1) SEG) in v (the whole warp calls): segment totals, a warp scan, then
// the lane whose segment holds the rank finds the bin.  -1 when the counts
// end at or before r; `before` gets the count below the bin, `in` its count.
template <int SEG>
__device__ __forceinline__ int warp_find_bin(const uint32_t (&v)[SEG], uint32_t r, uint32_t &before, uint32_t &in)
{
    const int lane = threadIdx.x & 31;
    const uint32_t c = segment_total(v);
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += x;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, incl > r);
    if (hit == 0u)
        return -1;
    const int L = __ffs(hit) - 1;
    int bin = -1;
    uint32_t b = 0, n = 0;
    if (lane == L)
        bin = lane * SEG + find_bin_in_segment(v, incl - c, r, b, n);
    before = __shfl_sync(0xffffffffu, b, L);
    in = __shfl_sync(0xffffffffu, n, L);
    return __shfl_sync(0xffffffffu, bin, L);
}

// Records that the counts disagree with the ranks (cannot happen with
// consistent counts): no record but NaNs, and TIM_ERR_BAD_INPUT.
__device__ __forceinline__ void counts_inconsistent(const MonArgs &a)
{
    atomicCAS(a.status, 0, static_cast<int>(TIM_ERR_BAD_INPUT));
    a.st->empty = 1;
}

// ---------------------------------------------------------------- the high digit
// The full pass's last CTA, warp j per target (lists mode): the high digit of
// the target's offset from the list's coarse then fine histogram (one round
// trip each) and the rank left inside that bin.
__device__ void select_high(const MonArgs &a)
{
    const int lane = threadIdx.x & 31, j = threadIdx.x >> 5, q = j >> 1;
    MonState *st = a.st;
    const uint32_t r = static_cast<uint32_t>(st->rank[j]);   // < count[q] <= cap < 2^31
    uint32_t v[8], before = 0, in = 0;
    load_segment<8>(a.hic + q * MON_COARSE + lane * 8, v);
    const int cb = warp_find_bin<8>(v, r, before, in);
    if (cb < 0) {
        if (lane == 0)
            counts_inconsistent(a);
        return;
    }
    const uint32_t r1 = r - before;
    load_segment<8>(a.hif + q * MON_FINE + cb * MON_COARSE + lane * 8, v);
    const int fb = warp_find_bin<8>(v, r1, before, in);
    if (lane == 0) {
        if (fb < 0) {
            counts_inconsistent(a);
        } else {
            st->prefix[j] = static_cast<uint32_t>(cb * MON_COARSE + fb);
            st->rank[j] = static_cast<long long>(r1 - before);
        }
    }
}

// ---------------------------------------------------------------- the record
// Thread 0: the batch record from the selected keys (st->prefix).
__device__ void write_record(const MonArgs &a)
{
    MonState *st = a.st;
    const unsigned long long n = __ldcg(&st->n_used), ne = __ldcg(&st->n_extreme);
    double *o = a.out;
    o[TIM_MON_N_USED] = static_cast<double>(n);
    o[TIM_MON_N_EXTREME] = static_cast<double>(ne);
    o[TIM_MON_FRAC_EXTREME] = n > 0 ? static_cast<double>(ne) / static_cast<double>(n) : 0.0;
    if (__ldcg(&st->empty)) {
        const double nan = __longlong_as_double(0x7ff8000000000000ll);
        o[TIM_MON_P95_ABS_DELTA] = o[TIM_MON_RATIO_Q01] = o[TIM_MON_RATIO_Q50] = o[TIM_MON_RATIO_Q99] = nan;
        return;
    }
    uint32_t key[MON_TARGETS];
    for (int t = 0; t < MON_TARGETS; ++t)
        key[t] = __ldcg(&st->prefix[t]);
    const double a0 = __uint_as_float(key[0]), a1 = __uint_as_float(key[1]);
    o[TIM_MON_P95_ABS_DELTA] = a0 + st->frac[0] * (a1 - a0);
    const int field[3] = {TIM_MON_RATIO_Q01, TIM_MON_RATIO_Q50, TIM_MON_RATIO_Q99};
    for (int i = 1; i < MON_QUANTILES; ++i) {
        const double r0 = expf(unkey_signed(key[2 * i]));
        const double r1 = expf(unkey_signed(key[2 * i + 1]));
        o[field[i - 1]] = r0 + st->frac[i] * (r1 - r0);
    }
}

// ---------------------------------------------------------------- selection over all tokens
// (When a bound missed or a list overflowed.)  Radix selection on the full
// 32-bit keys in three digit passes of 11, 11 and 10 bits.
template <int PASS>
constexpr int pass_bins() { return PASS == 3 ? MON_BINS3 : MON_BINS2; }

// Shared-memory histogram words of a pass: pass 1 counts delta's key only
// (|delta|'s bins follow from it), passes 2 and 3 keep one histogram per target.
template <int PASS>
constexpr int pass_smem_words() { return PASS == 1 ? MON_BINS1 : MON_TARGETS * pass_bins<PASS>(); }

// Does key k carry the digits that `prefix` fixed in the passes before PASS?
template <int PASS>
__device__ __forceinline__ bool in_prefix(uint32_t k, uint32_t prefix)
{
    if (PASS == 1)
        return true;
    const int s = digit_shift(PASS - 1, 32);
    return (k >> s) == (prefix >> s);
}

// One pass over all tokens into a shared-memory histogram (`sh`), added to
// the global one of the pass.
template <int PASS>
__device__ void all_token_pass(const MonArgs &a, uint32_t *sh)
{
    constexpr int NB = pass_bins<PASS>();
    zero_histogram<pass_smem_words<PASS>()>(sh);
    uint32_t pr[MON_TARGETS];   // in registers: the histogram atomics may alias shared memory
#pragma unroll
    for (int j = 0; j < MON_TARGETS; ++j)
        pr[j] = __ldcg(&a.st->prefix[j]);   // set by CTA 0 before the last grid barrier
    __syncthreads();
    for_token_groups<MON_UNROLL>(a, [&](int64_t, const float (&d)[4], const bool (&m)[4], const bool (&valid)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const bool used = valid[i] && usable(m[i], d[i]);
            const uint32_t kd = key_signed(d[i]);
            if (PASS == 1) {
                if (used)
                    atomicAdd(sh + (kd >> 21), 1u);
            } else {
                const uint32_t ka = key_abs(d[i]);
#pragma unroll
                for (int j = 0; j < MON_TARGETS; ++j) {
                    const uint32_t k = j < 2 ? ka : kd;
                    if (used && in_prefix<PASS>(k, pr[j]))
                        atomicAdd(sh + j * NB + digit_of<PASS>(k, 32), 1u);
                }
            }
        }
    });
    __syncthreads();
    flush_histogram<pass_smem_words<PASS>()>(sh, PASS == 1 ? a.hist1 : PASS == 2 ? a.hist2 : a.hist3);
}

// CTA of MON_TARGETS warps, warp j = target j: the digit of pass PASS that
// holds the target's rank (the prefix and rank updated).
template <int PASS>
__device__ void select_digit(const MonArgs &a)
{
    constexpr int NB = pass_bins<PASS>();
    constexpr int SEG = NB / 32;
    const int lane = threadIdx.x & 31, j = threadIdx.x >> 5;
    MonState *st = a.st;
    const uint32_t r = static_cast<uint32_t>(__ldcg(&st->rank[j]));   // < N < 2^31
    uint32_t before = 0, in = 0;
    int bin;
    if (PASS == 1 && j < 2) {   // |delta|'s 1024 bins from delta's 2048
        uint32_t v[32];
        load_abs_segment<32>(a.hist1, 1024, lane * 32, v);
        bin = warp_find_bin<32>(v, r, before, in);
    } else {
        const uint32_t *hg = PASS == 1 ? a.hist1 : PASS == 2 ? a.hist2 + j * NB : a.hist3 + j * NB;
        uint32_t v[SEG];
        load_segment<SEG>(hg + lane * SEG, v);
        bin = warp_find_bin<SEG>(v, r, before, in);
    }
    if (lane == 0) {
        if (bin < 0) {
            counts_inconsistent(a);
        } else {
            st->rank[j] = static_cast<long long>(r - before);
            st->prefix[j] = __ldcg(&st->prefix[j]) | (static_cast<uint32_t>(bin) << digit_shift(PASS, 32));
        }
    }
}

// Grid barrier of the selection pass (a cooperative launch: every CTA is
// resident).  Bounded: a CTA whose wait runs out records TIM_ERR_TIMEOUT and
// raises the call's abort word, on which every other waiting CTA leaves too.
__device__ bool grid_barrier(const MonArgs &a, unsigned &gen)
{
    __shared__ int ok_s;
    __syncthreads();
    if (threadIdx.x == 0) {
        MonState *st = a.st;
        __threadfence();
        atomicAdd(&st->barrier, 1u);
        const unsigned target = (gen + 1u) * gridDim.x;
        const uint64_t t0 = global_ns();
        bool ok = true;
        while (*reinterpret_cast<volatile unsigned *>(&st->barrier) < target) {
            if (*reinterpret_cast<volatile int *>(&st->abort)) {
                ok = false;
                break;
            }
            if (global_ns() - t0 > a.wait_budget_ns) {
                ok = false;
                atomicExch(&st->abort, 1);
                atomicCAS(a.status, 0, static_cast<int>(TIM_ERR_TIMEOUT));
                break;
            }
            __nanosleep(128);
        }
        __threadfence();
        ok_s = ok;
    }
    __syncthreads();
    ++gen;
    return ok_s != 0;
}

__device__ void select_over_all_tokens(const MonArgs &a, uint32_t *sh)
{
    unsigned gen = 0;
    all_token_pass<1>(a, sh);
    if (!grid_barrier(a, gen))
        return;
    if (blockIdx.x == 0)
        select_digit<1>(a);
    if (!grid_barrier(a, gen))
        return;
    all_token_pass<2>(a, sh);
    if (!grid_barrier(a, gen))
        return;
    if (blockIdx.x == 0)
        select_digit<2>(a);
    if (!grid_barrier(a, gen))
        return;
    all_token_pass<3>(a, sh);
    if (last_cta(&a.st->ticket[2])) {
        select_digit<3>(a);
        __syncthreads();
        if (threadIdx.x == 0)
            write_record(a);
    }
}

// ---------------------------------------------------------------- the selection pass (lists)
// Every list key whose offset has a target's high digit gives the target its
// low digit (offset bits below the high digit, at most 16), counted in the
// target's coarse (top 8 bits) and fine (all 16) low-digit histograms, lanes
// with equal digits added by one atomic.  (Appending the keys to a per-target
// buffer instead made ~2000 keys meet on one counter: 30 us of serialised
// atomics.)  When a quantile's two targets share their high bin, the second
// reads the first's histograms.  Then the last CTA, warp j per target, selects
// the low digit from the two histograms (one round trip each); the target's
// key is lo + (high << shift) + low.
// Counts low digit `low` of target j (a key in the target's high bin) in the
// target's two histograms, lanes with equal digits added by one atomic (a
// full warp calls; lanes with hit unset take no part).  Kept out of line: the
// gather loop stays small (it had been bound by instruction fetch).
__device__ __noinline__ void count_low_digit(const MonArgs &a, bool hit, int j, uint32_t low)
{
    const int lane = threadIdx.x & 31;
    const uint32_t tag = hit ? static_cast<uint32_t>(j) << 16 | low : 0xffffffffu;
    const unsigned same = __match_any_sync(0xffffffffu, tag);
    const unsigned same_c = __match_any_sync(0xffffffffu, hit ? tag >> 8 : 0xffffffffu);
    if (hit && lane == __ffs(same) - 1)
        atomicAdd(a.lof + static_cast<size_t>(j) * MON_FINE + low, static_cast<uint32_t>(__popc(same)));
    if (hit && lane == __ffs(same_c) - 1)
        atomicAdd(a.loc + j * MON_COARSE + (low >> 8), static_cast<uint32_t>(__popc(same_c)));
}

__device__ void select_in_lists(const MonArgs &a)
{
    __shared__ uint32_t lo_s[MON_QUANTILES], hd_s[MON_TARGETS];
    __shared__ int shift_s[MON_QUANTILES], dup_s[MON_TARGETS];
    __shared__ unsigned long long cnt_s[MON_QUANTILES];
    const int tid = threadIdx.x, lane = tid & 31;
    MonState *st = a.st;
    if (tid < MON_QUANTILES) {
        lo_s[tid] = st->lo[tid];
        shift_s[tid] = high_shift(st->span_bits[tid]);
        cnt_s[tid] = std::min<unsigned long long>(a.hot[tid * MON_HOT_STRIDE], a.cap);
    }
    if (tid < MON_TARGETS) {
        hd_s[tid] = st->prefix[tid];
        dup_s[tid] = (tid & 1) && st->prefix[tid] == st->prefix[tid - 1];
    }
    __syncthreads();
    // One list after another (the list's bound, shift and high digits stay in
    // registers), each grid-strided, kBatch keys per lane loaded before use;
    // the trip count is uniform over the warp (the vote needs every lane).
    // (The four lists as one index space, with fewer rounds of loads but each
    // key's list parameters read from shared memory, measured ~3 us slower.)
    constexpr int kBatch = 16;
    const uint32_t stride = gridDim.x * MON_THREADS;
    const uint64_t pol = l2_policy_evict_first();
    for (int q = 0; q < MON_QUANTILES; ++q) {
        const uint32_t n = static_cast<uint32_t>(cnt_s[q]);   // <= cap < 2^31
        const uint32_t lo = lo_s[q], hd0 = hd_s[2 * q], hd1 = hd_s[2 * q + 1];
        const int sh = shift_s[q];
        const bool dup1 = dup_s[2 * q + 1] != 0;
        const uint32_t *list = a.cand + static_cast<size_t>(q) * a.cap;
        for (uint32_t w0 = blockIdx.x * MON_THREADS + (tid & ~31); w0 < n; w0 += kBatch * stride) {
            uint32_t v[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const uint32_t i = w0 + lane + u * stride;
                v[u] = i < n ? ld_global_hint(list + i, pol) : 0u;   // demoted once read
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const bool in = w0 + lane + u * stride < n;
                const uint32_t x = v[u] - lo;
                const uint32_t hd = x >> sh;
                const bool h0 = in && hd == hd0, h1 = in && hd == hd1 && !dup1;
                if (__any_sync(0xffffffffu, h0 || h1)) {
                    const uint32_t low = x & ((1u << sh) - 1u);   // sh <= 16
                    count_low_digit(a, h0, 2 * q, low);
                    count_low_digit(a, h1, 2 * q + 1, low);
                }
            }
        }
    }
    uint32_t dup = 0;   // bit j: target j reads target j - 1's histograms
#pragma unroll
    for (int j = 0; j < MON_TARGETS; ++j)
        dup |= static_cast<uint32_t>(dup_s[j]) << j;
    if (!last_cta(&st->ticket[2]))
        return;
    // warp j: target j
    const int j = tid >> 5, q = j >> 1;
    const int src = ((dup >> j) & 1u) ? j - 1 : j;
    const int sh = shift_s[q];
    uint32_t r = static_cast<uint32_t>(__ldcg(&st->rank[j]));
    uint32_t low = 0, before = 0, in = 0;
    bool ok = true;
    if (sh > 0) {   // else the high digit is the whole offset
        uint32_t c8[8];
        load_segment<8>(a.loc + src * MON_COARSE + lane * 8, c8);
        const int cb = warp_find_bin<8>(c8, r, before, in);
        ok = cb >= 0;
        if (ok) {
            r -= before;
            load_segment<8>(a.lof + static_cast<size_t>(src) * MON_FINE + cb * MON_COARSE + lane * 8, c8);
            const int fb = warp_find_bin<8>(c8, r, before, in);
            ok = fb >= 0;
            low = static_cast<uint32_t>(cb * MON_COARSE + (fb < 0 ? 0 : fb));
        }
    }
    if (lane == 0) {
        if (!ok)
            counts_inconsistent(a);
        else
            st->prefix[j] = lo_s[q] + (hd_s[j] << sh) + low;
    }
    __syncthreads();
    if (tid == 0)
        write_record(a);
}

// ---------------------------------------------------------------- the selection kernel
constexpr int kSelCtasPerSm = 2;
constexpr size_t kSelSmem = 4 * MON_TARGETS * MON_BINS2;   // the all-token pass 2's histograms

__global__ void __launch_bounds__(MON_THREADS, kSelCtasPerSm) mon_select_kernel(const MonArgs a)
{
    extern __shared__ __align__(16) uint32_t sel_sh[];
    __shared__ int mode_s;   // 0 no used token (or inconsistent counts), 1 the lists, 2 all tokens
    pdl_wait();   // the full pass's results
    if (threadIdx.x == 0) {
        const MonState *st = a.st;
        mode_s = st->empty ? 0 : st->fallback ? 2 : 1;
    }
    __syncthreads();
    if (mode_s == 0) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            write_record(a);
    } else if (mode_s == 1) {
        select_in_lists(a);
    } else {
        select_over_all_tokens(a, sel_sh);
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

constexpr size_t kSampleSmem = 4 * SBD;

// Each kernel's dynamic shared memory.  (The largest shared-memory carveout
// as a hint made the call ~6 us slower.)
template <typename K>
cudaError_t smem_attributes(K kernel, size_t bytes)
{
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

int g_sel_ctas_per_sm = 0;   // resident selection CTAs per SM (a cooperative launch needs them all at once)

} // namespace

cudaError_t monitor_prepare_device()
{
    cudaError_t e = smem_attributes(mon_sample_kernel, kSampleSmem);
    if (e == cudaSuccess)
        e = smem_attributes(mon_scan_kernel, kScanSmem);
    if (e == cudaSuccess)
        e = smem_attributes(mon_select_kernel, kSelSmem);
    int per_sm = 0;
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mon_select_kernel, MON_THREADS, kSelSmem);
    if (e == cudaSuccess && per_sm < 1)
        e = cudaErrorInvalidConfiguration;
    g_sel_ctas_per_sm = std::min(per_sm, kSelCtasPerSm);
    return e;
}

// memset of the state and small histograms, then the sample (+ bounds), the
// full pass (+ ranks and high digits) chained by dependent launches, and the
// selection pass (a cooperative launch: its all-token mode has grid barriers).
cudaError_t monitor_launch(const MonArgs &a, int num_sms, cudaStream_t stream)
{
    cudaError_t e = cudaMemsetAsync(a.st, 0, MON_ZEROED_BYTES, stream);
    if (e != cudaSuccess)
        return e;
    const int64_t groups = (a.N + 3) / 4;
    const int64_t want = (groups + kScanThreads - 1) / kScanThreads;
    const dim3 scan_grid(static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(want, num_sms))));
    // one CTA per SM: all start at once; every one of them also zeroes its
    // share of the fine histograms
    const dim3 block(MON_THREADS);
    if ((e = launch_pdl(mon_sample_kernel, dim3(static_cast<unsigned>(num_sms)), block, kSampleSmem, stream, a)) !=
            cudaSuccess ||
        (e = launch_pdl(mon_scan_kernel, scan_grid, dim3(kScanThreads), kScanSmem, stream, a)) != cudaSuccess)
        return e;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1] = pdl_attribute();
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cfg.gridDim = dim3(static_cast<unsigned>(std::max(1, g_sel_ctas_per_sm) * num_sms));
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = kSelSmem;
    return cudaLaunchKernelEx(&cfg, mon_select_kernel, a);
}

} // namespace tim
