// monitor_internal.h -- launch parameters of the mismatch monitor (exact quantiles by selection).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace tim {

constexpr int MON_THREADS = 256;
constexpr int MON_UNROLL = 4;          // 4-token groups per thread per iteration, loaded before use
constexpr int MON_QUANTILES = 4;       // p95 |delta|; ratio 0.01, 0.5, 0.99
constexpr int MON_TARGETS = 8;         // order statistics: ranks k and k + 1 of each quantile
constexpr int MON_BINS1 = 2048;        // selection over all tokens: digit 1, 11 key bits
constexpr int MON_BINS2 = 2048;        // digit 2: 11 bits
constexpr int MON_BINS3 = 1024;        // digit 3: 10 bits
constexpr int MON_SAMPLE_RUNS = 1024;  // the sample: up to 1024 runs of MON_SAMPLE_RUN consecutive tokens
constexpr int MON_SAMPLE_RUN = 1024;
constexpr int MON_SBINS = 16384;       // sample histogram of delta's key >> 18 (|delta|'s follows from it)
// Collected keys: the offset key - lo of a quantile's list splits into a high
// digit (its top 16 bits) and a low one (the rest, at most 16 bits).  The full
// pass counts the high digits, the selection pass, per target, the low digits
// of the keys in the target's high bin: each in a coarse histogram (the top 8
// bits of the digit) and a fine one (all 16).
constexpr int MON_HI_BITS = 16;
constexpr int MON_FINE = 1 << MON_HI_BITS;   // 65536 bins
constexpr int MON_COARSE = 256;              // bins of the top 8 bits of a 16-bit digit

// Device state of one call, at the start of the workspace (zeroed before the sample).
struct MonState {
    unsigned long long n_used, n_extreme, sample_used;
    unsigned long long below[MON_QUANTILES];   // used tokens with key < lo
    long long rank[MON_TARGETS];               // rank still to find inside the current prefix
    uint32_t lo[MON_QUANTILES], hi[MON_QUANTILES];
    uint32_t prefix[MON_TARGETS];              // all tokens: the key bits fixed so far; lists: the high digit;
                                               // at the end, the selected key
    int span_bits[MON_QUANTILES];              // lists: bit length of hi - lo
    double frac[MON_QUANTILES];                // interpolation weight of each quantile
    int empty;                                 // no used token
    int fallback;                              // 1: select over all tokens (a bound missed)
    unsigned ticket[3];                        // CTAs finished: sample, full pass, selection pass
    unsigned barrier;                          // the selection pass's grid barrier (all-token mode)
    int abort;                                 // a grid-barrier wait ran out: every CTA leaves
};

// The lists' lengths, which every warp of the full pass reserves room from,
// each in its own 256-byte line after the state (atomics on one line are
// served one after another): word MON_HOT_STRIDE q = used tokens with lo <=
// key <= hi of quantile q (the list's length, kept up to cap).
constexpr int MON_HOT_STRIDE = 32;   // 8-byte words: 256 bytes

// Workspace (all offsets 256-byte aligned):
//   zeroed per call by a memset: the state, the all-token histograms (digits
//   1..3), the sample histogram, the lists' coarse histograms and the targets'
//   coarse low-digit histograms;
//   zeroed per call by the sample kernel: the lists' fine histograms and the
//   targets' fine low-digit histograms (3 MB);
//   then the four candidate lists of `cap` keys.
constexpr size_t MON_STATE_BYTES = 2048;   // the state (512 bytes), then the hot counters
static_assert(sizeof(MonState) <= 512 && 512 + 8 * MON_HOT_STRIDE * MON_QUANTILES <= MON_STATE_BYTES,
              "state block");
constexpr size_t MON_HIST1_WORDS = MON_BINS1;
constexpr size_t MON_HIST2_WORDS = MON_TARGETS * MON_BINS2;
constexpr size_t MON_HIST3_WORDS = MON_TARGETS * MON_BINS3;
constexpr size_t MON_SHIST_WORDS = MON_SBINS;
constexpr size_t MON_HIC_WORDS = MON_QUANTILES * MON_COARSE;
constexpr size_t MON_LOC_WORDS = MON_TARGETS * MON_COARSE;
constexpr size_t MON_ZEROED_BYTES =
    MON_STATE_BYTES + 4 * (MON_HIST1_WORDS + MON_HIST2_WORDS + MON_HIST3_WORDS + MON_SHIST_WORDS + MON_HIC_WORDS +
                           MON_LOC_WORDS);
constexpr size_t MON_HIF_WORDS = static_cast<size_t>(MON_QUANTILES) * MON_FINE;
constexpr size_t MON_LOF_WORDS = static_cast<size_t>(MON_TARGETS) * MON_FINE;
static_assert(MON_ZEROED_BYTES % 256 == 0, "aligned regions");

inline unsigned long long monitor_cap(int64_t N) { return static_cast<unsigned long long>(N / 16 + 65536); }
inline size_t monitor_workspace_bytes(int64_t N)
{
    return MON_ZEROED_BYTES + 4 * (MON_HIF_WORDS + MON_LOF_WORDS) +
           4ull * MON_QUANTILES * monitor_cap(N);
}

struct MonArgs {
    const float *l_tr, *l_ro;
    const uint8_t *mask;
    int64_t N;
    float tau_tok;
    uint8_t *reject;     // optional [N]
    double *out;         // [TIM_MON_FIELDS]
    MonState *st;
    unsigned long long *hot;           // [MON_QUANTILES][MON_HOT_STRIDE]: the lists' lengths
    uint32_t *hist1, *hist2, *hist3;   // selection over all tokens: [MON_BINS1], [8][MON_BINS2], [8][MON_BINS3]
    uint32_t *shist;     // sample histogram of delta's key [MON_SBINS]
    uint32_t *hic, *hif; // lists' high digits: coarse [4][MON_COARSE], fine [4][MON_FINE]
    uint32_t *loc, *lof; // targets' low digits: coarse [8][MON_COARSE], fine [8][MON_FINE]
    uint32_t *cand;      // [MON_QUANTILES][cap] collected keys
    unsigned long long cap;
    int *status;
    uint64_t wait_budget_ns;   // bound of each pipeline wait in the kernels
};

// Points the arrays of `a` into a workspace of monitor_workspace_bytes(N) bytes.
inline void monitor_bind(MonArgs &a, void *ws, int64_t N)
{
    char *p = static_cast<char *>(ws);
    a.st = reinterpret_cast<MonState *>(p);
    a.hot = reinterpret_cast<unsigned long long *>(p + 512);
    a.hist1 = reinterpret_cast<uint32_t *>(p + MON_STATE_BYTES);
    a.hist2 = a.hist1 + MON_HIST1_WORDS;
    a.hist3 = a.hist2 + MON_HIST2_WORDS;
    a.shist = a.hist3 + MON_HIST3_WORDS;
    a.hic = a.shist + MON_SHIST_WORDS;
    a.loc = a.hic + MON_HIC_WORDS;
    a.hif = a.loc + MON_LOC_WORDS;
    a.lof = a.hif + MON_HIF_WORDS;
    a.cand = a.lof + MON_LOF_WORDS;
    a.cap = monitor_cap(N);
}

cudaError_t monitor_launch(const MonArgs &a, int num_sms, cudaStream_t stream);
cudaError_t monitor_prepare_device();

} // namespace tim
