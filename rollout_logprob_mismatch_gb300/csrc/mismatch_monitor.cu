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
//   mon_sample_kernel   histograms (14 key bits) of up to 1024 evenly spaced
//                       runs of 1024 consecutive tokens;
//   mon_bounds_kernel   per quantile, key bounds [lo, hi] around the sample's
//                       quantile, six standard deviations of its rank wide;
//   mon_scan_kernel     the one full pass (bulk-copied chunks): n_used,
//                       n_extreme, rejection flags and, per quantile, the used
//                       tokens below lo and the keys inside [lo, hi]
//                       (typically a few percent), kept in a list;
//   mon_check_kernel    ranks from n_used; each quantile's order statistics
//                       must fall inside its list (else, or if a list
//                       overflowed, the selection runs over all tokens);
//   mon_pass_kernel<1..3> + mon_select_kernel<1..3>: radix selection in three
//                       digit passes (11, 11, 10 bits) over the lists, on
//                       key - lo, or over all tokens; select<3> writes the
//                       record.
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
static_assert(SBD + SBA <= MON_SBINS_D + MON_SBINS_A, "sample histogram room");
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

// ---------------------------------------------------------------- sample
// Run r: tokens [s, s + MON_SAMPLE_RUN), s = r N / runs (runs back to back
// when they cover the batch); CTA c takes runs c, c + gridDim, ... into
// shared-memory histograms and adds the non-zero bins to the global ones.
__global__ void __launch_bounds__(MON_THREADS) mon_sample_kernel(const MonArgs a)
{
    extern __shared__ __align__(16) uint32_t sh[];   // [SBD] delta, then [SBA] |delta|
    const int tid = threadIdx.x, lane = tid & 31;
    for (int i = tid; i < SBD + SBA; i += MON_THREADS)
        sh[i] = 0u;
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();
    const int64_t N = a.N;
    const int64_t cover = static_cast<int64_t>(MON_SAMPLE_RUNS) * MON_SAMPLE_RUN;
    const int64_t runs = std::min<int64_t>(MON_SAMPLE_RUNS, (N + MON_SAMPLE_RUN - 1) / MON_SAMPLE_RUN);
    int used = 0;
    for (int64_t r = blockIdx.x; r < runs; r += gridDim.x) {
        const int64_t s0 = N <= cover ? r * MON_SAMPLE_RUN : r * N / runs;
        const int64_t s1 = std::min<int64_t>(N, s0 + MON_SAMPLE_RUN);
        for (int64_t t = s0 + tid; t < s1; t += MON_THREADS) {
            const float d = delta_of(a.l_tr[t], a.l_ro[t]);
            if (usable(a.mask[t] != 0, d)) {
                atomicAdd(sh + (key_signed(d) >> SAMPLE_SHIFT), 1u);
                atomicAdd(sh + SBD + (key_abs(d) >> SAMPLE_SHIFT), 1u);
                ++used;
            }
        }
    }
    used = __reduce_add_sync(0xffffffffu, used);
    if (lane == 0 && used)
        atomicAdd(&a.st->sample_used, static_cast<unsigned long long>(used));
    __syncthreads();
    for (int i = tid; i < SBD + SBA; i += MON_THREADS)
        if (sh[i] != 0u)
            atomicAdd(a.shist + i, sh[i]);
}

// ---------------------------------------------------------------- bounds
// One CTA of 1024 threads.  For quantile q at level L with m sampled used
// tokens: sample ranks floor(L (m - 1)) - w and ceil(L (m - 1)) + w, w = six
// standard deviations of a sample quantile's rank (sqrt(m L (1 - L))) + 2;
// lo = the lowest key of the bin holding the first (0 when that rank is at or
// below the sample's first), hi = the highest key of the bin holding the
// second (all ones when at or above the sample's last).
__global__ void __launch_bounds__(1024) mon_bounds_kernel(const MonArgs a)
{
    extern __shared__ __align__(16) uint32_t hs[];   // the sample histograms, copied with coalesced loads
    __shared__ long long wsum[32];
    __shared__ int bin_s[2 * MON_QUANTILES];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    pdl_launch_dependents();
    MonState *st = a.st;
    __shared__ long long rlo_s[MON_QUANTILES], rhi_s[MON_QUANTILES];
    const long long m = static_cast<long long>(st->sample_used);
    if (tid < MON_QUANTILES) {   // fp64 in a few threads only: GB300 runs it slowly
        const double L = level(tid);
        const double j = static_cast<double>(m - 1) * L;
        const long long w = static_cast<long long>(ceil(kSigmas * sqrt(static_cast<double>(m) * L * (1.0 - L)))) + 2;
        rlo_s[tid] = static_cast<long long>(floor(j)) - w;
        rhi_s[tid] = static_cast<long long>(ceil(j)) + w;
    }
    if (tid < 2 * MON_QUANTILES)
        bin_s[tid] = -1;
#pragma unroll 24
    for (int i = tid; i < SBD + SBA; i += 1024)
        hs[i] = a.shist[i];
    __syncthreads();
    for (int kind = 0; kind < 2; ++kind) {   // 0: delta (quantiles 1..3), 1: |delta| (quantile 0)
        const int nb = kind == 0 ? SBD : SBA;
        const uint32_t *h = hs + (kind == 0 ? 0 : SBD);
        const int per = nb / 1024;
        long long c = 0;
        for (int b = 0; b < per; ++b)
            c += h[tid * per + b];
        long long incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += v;
        }
        __syncthreads();   // the previous kind's wsum reads are done
        if (lane == 31)
            wsum[warp] = incl;
        __syncthreads();
        long long before_warp = 0;
        for (int w = 0; w < warp; ++w)
            before_warp += wsum[w];
        const long long excl = before_warp + incl - c;
        const int q_first = kind == 0 ? 1 : 0, q_end = kind == 0 ? MON_QUANTILES : 1;
        for (int q = q_first; q < q_end; ++q) {
            for (int e = 0; e < 2; ++e) {
                const long long R = e == 0 ? rlo_s[q] : rhi_s[q];
                if (m > 0 && R > 0 && R < m - 1 && excl <= R && R < excl + c) {
                    long long cum = excl;
                    for (int b = 0; b < per; ++b) {
                        cum += h[tid * per + b];
                        if (cum > R) {
                            bin_s[2 * q + e] = tid * per + b;
                            break;
                        }
                    }
                }
            }
        }
    }
    __syncthreads();
    if (tid < MON_QUANTILES) {
        const int q = tid;
        const int bl = bin_s[2 * q], bh = bin_s[2 * q + 1];
        st->lo[q] = bl < 0 ? 0u : static_cast<uint32_t>(bl) << SAMPLE_SHIFT;
        st->hi[q] = bh < 0 ? 0xffffffffu : (static_cast<uint32_t>(bh) << SAMPLE_SHIFT) | ((1u << SAMPLE_SHIFT) - 1u);
    }
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
constexpr int kScanWarps = MON_THREADS / 32;
constexpr int kScanCtasPerSm = 2;                       // the rings and stages: 82 KB of shared memory per CTA
constexpr size_t kRingBytes = static_cast<size_t>(kScanWarps) * kRing * kChunkBytes;
constexpr size_t kStageBytes = sizeof(uint32_t) * kScanWarps * MON_QUANTILES * kStage;
constexpr size_t kScanSmem = kRingBytes + kStageBytes + 8 * kScanWarps * kRing;
static_assert(kChunkF % 16 == 0 && kChunkBytes % 16 == 0 && kRingBytes % 16 == 0, "bulk copies stay 16-byte aligned");

__device__ __forceinline__ void flush_stage(const MonArgs &a, const uint32_t *buf, int q, int n, int lane)
{
    unsigned long long base = 0;
    if (lane == 0)
        base = atomicAdd(&a.st->count[q], static_cast<unsigned long long>(n));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (lane < n && base + lane < a.cap)
        a.cand[static_cast<size_t>(q) * a.cap + base + lane] = buf[lane];
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

__global__ void __launch_bounds__(MON_THREADS, kScanCtasPerSm) mon_scan_kernel(const MonArgs a)
{
    extern __shared__ __align__(16) uint8_t scan_smem[];   // rings [warp][kRing], staging, barriers
    __shared__ float flo_s[MON_QUANTILES], fhi_s[MON_QUANTILES];
    __shared__ uint32_t one_s;
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
    pdl_wait();
    pdl_launch_dependents();
    if (tid < MON_QUANTILES) {
        const uint32_t lo = a.st->lo[tid], hi = a.st->hi[tid];
        flo_s[tid] = tid == 0 ? abs_lo_threshold(lo) : signed_lo_threshold(lo);
        fhi_s[tid] = tid == 0 ? abs_hi_threshold(hi) : signed_hi_threshold(hi);
    }
    __syncthreads();
    float flo[MON_QUANTILES], fhi[MON_QUANTILES];
#pragma unroll
    for (int q = 0; q < MON_QUANTILES; ++q) {
        flo[q] = flo_s[q];
        fhi[q] = fhi_s[q];
    }
    const uint32_t one = one_s;
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

    // The warp's k-th chunk: groups [c_k kChunk, (c_k + 1) kChunk), c_k = w + k warps.
    const int64_t w = static_cast<int64_t>(blockIdx.x) * kScanWarps + warp;
    auto whole = [&](int64_t k) { return (w + k * warps + 1) * kChunk <= full; };
    auto issue = [&](int64_t k) {   // lane 0: stage chunk k into ring slot k % kRing
        if (lane != 0 || !whole(k))
            return;
        const int64_t g0 = (w + k * warps) * kChunk;
        const int slot = static_cast<int>(k % kRing);
        const uint32_t dst = smem_u32(ring + slot * kChunkBytes), bar = bar0 + 8u * slot;
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
                    base = atomicAdd(&a.st->count[q], static_cast<unsigned long long>(total));
                base = __shfl_sync(0xffffffffu, base, 0) + static_cast<unsigned long long>(excl);
                for (uint32_t b = inbits[q]; b != 0u; b &= b - 1u, ++base) {
                    const float v = pick(dv, __ffs(b) - 1);
                    if (base < a.cap)
                        a.cand[static_cast<size_t>(q) * a.cap + base] = q == 0 ? key_abs(v) : key_signed(v);
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
                flush_stage(a, buf, q, 32, lane);
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
    for (int k = 0; k < kRing; ++k)
        issue(k);
    bool ok = true;
    int64_t k = 0;
    for (; whole(k); ++k) {
        const int slot = static_cast<int>(k % kRing);
        if (!mbar_wait_sleep(bar0 + 8u * slot, static_cast<uint32_t>((k / kRing) & 1), abort_flag,
                             a.wait_budget_ns)) {
            ok = false;
            break;
        }
        step((w + k * warps) * kChunk, ring + slot * kChunkBytes, std::false_type{});
        __syncwarp();   // every lane has read the slot
        issue(k + kRing);
    }
    if (!ok) {   // copies may still be landing: let them, then report
        for (int64_t j = k; j < k + kRing; ++j)
            if (whole(j))
                drain_wait(bar0 + 8u * static_cast<uint32_t>(j % kRing), static_cast<uint32_t>((j / kRing) & 1));
        if (lane == 0)
            atomicCAS(a.status, 0, static_cast<int>(TIM_ERR_TIMEOUT));
        return;
    }
    if ((w + k * warps) * kChunk < G)
        step((w + k * warps) * kChunk, nullptr, std::true_type{});

    __syncwarp();
#pragma unroll
    for (int q = 0; q < MON_QUANTILES; ++q)
        if (staged[q] > 0)
            flush_stage(a, stage_all + (warp * MON_QUANTILES + q) * kStage, q, staged[q], lane);
    const int wu = __reduce_add_sync(0xffffffffu, n_used);
    const int we = __reduce_add_sync(0xffffffffu, n_ext);
    int wb[MON_QUANTILES];
#pragma unroll
    for (int q = 0; q < MON_QUANTILES; ++q)
        wb[q] = __reduce_add_sync(0xffffffffu, n_used - at_or_above[q]);
    if (lane == 0) {
        atomicAdd(&a.st->n_used, static_cast<unsigned long long>(wu));
        atomicAdd(&a.st->n_extreme, static_cast<unsigned long long>(we));
#pragma unroll
        for (int q = 0; q < MON_QUANTILES; ++q)
            if (wb[q])
                atomicAdd(&a.st->below[q], static_cast<unsigned long long>(wb[q]));
    }
}

// ---------------------------------------------------------------- ranks and mode
__global__ void mon_check_kernel(const MonArgs a)
{
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x != 0)
        return;
    MonState *st = a.st;
    const long long n = static_cast<long long>(st->n_used);
    st->empty = n == 0;
    if (n == 0)
        return;
    bool ok = true;
    long long k[MON_QUANTILES], k1[MON_QUANTILES];
    for (int q = 0; q < MON_QUANTILES; ++q) {
        const double h = static_cast<double>(n - 1) * level(q);
        const double fl = floor(h);
        k[q] = static_cast<long long>(fl);
        k1[q] = k[q] + 1 < n ? k[q] + 1 : k[q];
        st->frac[q] = h - fl;
        const long long b = static_cast<long long>(st->below[q]);
        const long long c = static_cast<long long>(st->count[q]);
        ok = ok && c <= static_cast<long long>(a.cap) && b <= k[q] && k1[q] < b + c;
    }
    st->fallback = ok ? 0 : 1;
    for (int q = 0; q < MON_QUANTILES; ++q) {
        const long long b = ok ? static_cast<long long>(st->below[q]) : 0;
        st->rank[2 * q] = k[q] - b;
        st->rank[2 * q + 1] = k1[q] - b;
        const uint32_t span = st->hi[q] - st->lo[q];
        st->span_bits[q] = ok ? (span == 0u ? 0 : 32 - __clz(static_cast<int>(span))) : 32;
    }
}

// ---------------------------------------------------------------- radix passes
// Digits of a value with b significant bits (b = 32 for raw keys): pass 1 the
// top 11 (bits b-11 .. b-1), pass 2 the next 11, pass 3 the rest (<= 10).
__device__ __forceinline__ int digit_shift(int pass, int b)
{
    return pass == 1 ? max(b - 11, 0) : pass == 2 ? max(b - 22, 0) : 0;
}

template <int PASS>
constexpr int pass_bins() { return PASS == 3 ? MON_BINS3 : MON_BINS2; }

template <int PASS>
constexpr int pass_smem_words()
{
    return PASS == 1 ? MON_QUANTILES * MON_BINS1 : MON_TARGETS * pass_bins<PASS>();
}

// Does v carry the digits that `prefix` fixed in the passes before PASS?
template <int PASS>
__device__ __forceinline__ bool in_prefix(uint32_t v, uint32_t prefix, int b)
{
    if (PASS == 1)
        return true;
    const int s = digit_shift(PASS - 1, b);
    return (static_cast<uint64_t>(v) >> s) == (static_cast<uint64_t>(prefix) >> s);
}

template <int PASS>
__device__ __forceinline__ uint32_t digit_of(uint32_t v, int b)
{
    const int s = digit_shift(PASS, b);
    const int top = PASS == 1 ? b : digit_shift(PASS - 1, b);
    const int width = top - s;   // <= 11
    return (v >> s) & ((1u << width) - 1u);
}

template <int PASS>
__global__ void __launch_bounds__(MON_THREADS, MON_CTAS_PER_SM) mon_pass_kernel(const MonArgs a)
{
    constexpr int NB = pass_bins<PASS>();
    extern __shared__ __align__(16) uint32_t mon_sh[];
    __shared__ uint32_t pref_s[MON_TARGETS], lo_s[MON_QUANTILES];
    __shared__ int bits_s[MON_QUANTILES];
    __shared__ int mode_s;   // 0 nothing to do, 1 the collected lists, 2 all tokens
    __shared__ unsigned long long cnt_s[MON_QUANTILES];
    const int tid = threadIdx.x;
    pdl_wait();
    pdl_launch_dependents();
    MonState *st = a.st;
    if (tid < MON_TARGETS)
        pref_s[tid] = st->prefix[tid];
    if (tid < MON_QUANTILES) {
        lo_s[tid] = st->lo[tid];
        bits_s[tid] = st->span_bits[tid];
        cnt_s[tid] = std::min<unsigned long long>(st->count[tid], a.cap);
    }
    if (tid == 0)
        mode_s = st->empty ? 0 : st->fallback ? 2 : 1;
    __syncthreads();
    const unsigned long long total = cnt_s[0] + cnt_s[1] + cnt_s[2] + cnt_s[3];
    // Collected keys: at least kKeysPerCta per CTA, so that few CTAs pay for
    // clearing and adding their histograms; the others leave at once.
    constexpr unsigned long long kKeysPerCta = 16 * MON_THREADS;
    const unsigned long long ctas = std::min<unsigned long long>(gridDim.x, (total + kKeysPerCta - 1) / kKeysPerCta);
    // uniform over the CTA: nothing to select, or no collected key for this CTA
    if (mode_s == 0 || (mode_s == 1 && blockIdx.x >= ctas))
        return;
    for (int i = tid; i < pass_smem_words<PASS>(); i += MON_THREADS)
        mon_sh[i] = 0u;
    __syncthreads();
    if (mode_s == 1) {
        // the collected keys of the four lists, one list after another
        for (unsigned long long i = static_cast<unsigned long long>(blockIdx.x) * MON_THREADS + tid; i < total;
             i += ctas * MON_THREADS) {
            int q = 0;
            unsigned long long off = i;
            while (off >= cnt_s[q]) {   // ends at q <= 3 because i < total
                off -= cnt_s[q];
                ++q;
            }
            const uint32_t v = a.cand[static_cast<size_t>(q) * a.cap + off] - lo_s[q];
            const int b = bits_s[q];
            if (PASS == 1) {
                atomicAdd(mon_sh + q * MON_BINS1 + digit_of<1>(v, b), 1u);
            } else {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int j = 2 * q + e;
                    if (in_prefix<PASS>(v, pref_s[j], b))
                        atomicAdd(mon_sh + j * NB + digit_of<PASS>(v, b), 1u);
                }
            }
        }
    } else {
        uint32_t pr[MON_TARGETS];   // in registers: the histogram atomics may alias shared memory
#pragma unroll
        for (int j = 0; j < MON_TARGETS; ++j)
            pr[j] = pref_s[j];
        for_token_groups<MON_UNROLL>(a, [&](int64_t, const float (&d)[4], const bool (&m)[4], const bool (&valid)[4]) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const bool used = valid[i] && usable(m[i], d[i]);
                const uint32_t kd = key_signed(d[i]);
                if (PASS == 1) {
                    if (used)   // delta's key only; |delta|'s histogram follows (mon_select_kernel<1>)
                        atomicAdd(mon_sh + (kd >> 21), 1u);
                } else {
                    const uint32_t ka = key_abs(d[i]);
#pragma unroll
                    for (int j = 0; j < MON_TARGETS; ++j) {
                        const uint32_t k = j < 2 ? ka : kd;
                        if (used && in_prefix<PASS>(k, pr[j], 32))
                            atomicAdd(mon_sh + j * NB + digit_of<PASS>(k, 32), 1u);
                    }
                }
            }
        });
    }
    __syncthreads();
    uint32_t *gh = PASS == 1 ? a.hist1 : PASS == 2 ? a.hist2 : a.hist3;
    for (int i = tid; i < pass_smem_words<PASS>(); i += MON_THREADS) {
        const uint32_t c = mon_sh[i];
        if (c != 0u)
            atomicAdd(gh + i, c);
    }
}

// Per target (warp j): the bin of pass PASS that holds the target's rank, and
// the rank left inside it; PASS 3 then writes the record.  One CTA of
// MON_TARGETS warps.
template <int PASS>
__global__ void __launch_bounds__(MON_TARGETS * 32) mon_select_kernel(const MonArgs a)
{
    constexpr int NB = pass_bins<PASS>();
    extern __shared__ __align__(16) uint32_t hist_s[];   // each warp's histogram, copied with coalesced loads
    const int tid = threadIdx.x, lane = tid & 31, j = tid >> 5, q = j >> 1;
    MonState *st = a.st;
    pdl_wait();
    pdl_launch_dependents();
    if (!st->empty) {
        const bool all_tokens = st->fallback != 0;
        const int b = all_tokens ? 32 : st->span_bits[q];
        // The all-token pass 1 counted delta's key only.  |delta| has a clear
        // top bit, and its bin c holds the positive deltas of delta-bin
        // 1024 + c and the negative ones of delta-bin 1023 - c.
        const bool abs1 = PASS == 1 && all_tokens && j < 2;
        const uint32_t *hg = PASS == 1 ? a.hist1 + (all_tokens ? 0 : q * MON_BINS1)
                           : PASS == 2 ? a.hist2 + j * NB
                                       : a.hist3 + j * NB;
        uint32_t *h = hist_s + j * 2048;
#pragma unroll 16
        for (int x = lane; x < NB; x += 32)
            h[x] = hg[x];
        __syncwarp();
        auto count = [&](int c) -> long long {
            return abs1 ? static_cast<long long>(h[1024 + c]) + h[1023 - c] : static_cast<long long>(h[c]);
        };
        const long long r = st->rank[j];
        const int SEG = (abs1 ? 1024 : NB) / 32;   // bins per lane
        long long c = 0;
        for (int x = 0; x < SEG; ++x)
            c += count(lane * SEG + x);
        long long incl = c;
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
                for (int x = 0; x < SEG; ++x) {
                    const long long hb = count(lane * SEG + x);
                    if (cum + hb > r) {
                        bin = lane * SEG + x;
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
                st->prefix[j] |= static_cast<uint32_t>(bin) << digit_shift(PASS, b);
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
    uint32_t key[MON_TARGETS];
    for (int t = 0; t < MON_TARGETS; ++t)
        key[t] = st->fallback ? st->prefix[t] : st->lo[t >> 1] + st->prefix[t];
    const double a0 = __uint_as_float(key[0]), a1 = __uint_as_float(key[1]);
    o[TIM_MON_P95_ABS_DELTA] = a0 + st->frac[0] * (a1 - a0);
    const int field[3] = {TIM_MON_RATIO_Q01, TIM_MON_RATIO_Q50, TIM_MON_RATIO_Q99};
    for (int i = 1; i < MON_QUANTILES; ++i) {
        const double r0 = expf(unkey_signed(key[2 * i]));
        const double r1 = expf(unkey_signed(key[2 * i + 1]));
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

constexpr size_t kSampleSmem = 4 * (SBD + SBA);
constexpr size_t kSelectSmem = 4 * MON_TARGETS * 2048;

} // namespace

cudaError_t monitor_prepare_device()
{
    cudaError_t e = cudaFuncSetAttribute(mon_sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSampleSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mon_bounds_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSampleSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mon_select_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSelectSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mon_select_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSelectSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mon_select_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSelectSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mon_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kScanSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mon_pass_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 4 * pass_smem_words<1>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mon_pass_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 4 * pass_smem_words<2>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mon_pass_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 4 * pass_smem_words<3>());
    return e;
}

cudaError_t monitor_launch(const MonArgs &a, int num_sms, cudaStream_t stream)
{
    cudaError_t e = cudaMemsetAsync(a.st, 0, MON_ZEROED_BYTES, stream);
    if (e != cudaSuccess)
        return e;
    const int64_t groups = (a.N + 3) / 4;
    const int64_t want = (groups + MON_THREADS - 1) / MON_THREADS;
    const dim3 grid(static_cast<unsigned>(
        std::max<int64_t>(1, std::min<int64_t>(want, static_cast<int64_t>(MON_CTAS_PER_SM) * num_sms))));
    const int64_t scan_want = (groups + (MON_THREADS / 32) * 32 * kScanGroups - 1) / ((MON_THREADS / 32) * 32 * kScanGroups);
    const dim3 scan_grid(static_cast<unsigned>(
        std::max<int64_t>(1, std::min<int64_t>(scan_want, static_cast<int64_t>(kScanCtasPerSm) * num_sms))));
    const int64_t runs = std::max<int64_t>(
        1, std::min<int64_t>({static_cast<int64_t>(MON_SAMPLE_RUNS), (a.N + MON_SAMPLE_RUN - 1) / MON_SAMPLE_RUN,
                              2LL * num_sms}));
    const dim3 block(MON_THREADS), sel(MON_TARGETS * 32);
    if ((e = launch_pdl(mon_sample_kernel, dim3(static_cast<unsigned>(runs)), block, kSampleSmem, stream, a)) !=
            cudaSuccess ||
        (e = launch_pdl(mon_bounds_kernel, dim3(1), dim3(1024), kSampleSmem, stream, a)) != cudaSuccess ||
        (e = launch_pdl(mon_scan_kernel, scan_grid, block, kScanSmem, stream, a)) != cudaSuccess ||
        (e = launch_pdl(mon_check_kernel, dim3(1), dim3(32), 0, stream, a)) != cudaSuccess ||
        (e = launch_pdl(mon_pass_kernel<1>, grid, block, 4 * pass_smem_words<1>(), stream, a)) != cudaSuccess ||
        (e = launch_pdl(mon_select_kernel<1>, dim3(1), sel, kSelectSmem, stream, a)) != cudaSuccess ||
        (e = launch_pdl(mon_pass_kernel<2>, grid, block, 4 * pass_smem_words<2>(), stream, a)) != cudaSuccess ||
        (e = launch_pdl(mon_select_kernel<2>, dim3(1), sel, kSelectSmem, stream, a)) != cudaSuccess ||
        (e = launch_pdl(mon_pass_kernel<3>, grid, block, 4 * pass_smem_words<3>(), stream, a)) != cudaSuccess)
        return e;
    return launch_pdl(mon_select_kernel<3>, dim3(1), sel, kSelectSmem, stream, a);
}

} // namespace tim
