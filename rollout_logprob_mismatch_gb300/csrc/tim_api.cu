// tim_api.cu -- the C ABI declared in include/tim.h: argument checks, per-device
// set-up (sm_103 check, memory pool, tensor-map encoder), workspace, launches.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/tim.h"
#include "bwd_internal.h"
#include "monitor_internal.h"
#include "ppo_internal.h"
#include "k1_internal.h"
#include "k2_internal.h"
#include "tim_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kVersion = 100;   // 0.1.0

thread_local char g_msg[512] = "";

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(TIM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Status block written by the kernels of this library: the status (first error
// wins) and, in the checked build, the first violation (tim::STATUS_WORDS).
__device__ __align__(16) int g_status[tim::STATUS_WORDS];

struct DeviceState {
    bool ready = false;
    int status_code = TIM_OK;   // why the device is unusable, if it is
    int sms = 0;
    int *status = nullptr;      // device address of g_status
    cudaMemPool_t pool = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

uint64_t wait_budget_ns()
{
    static const uint64_t v = [] {
        const char *s = std::getenv("TIM_WAIT_BUDGET_MS");
        const long long ms = s ? std::atoll(s) : 0;
        return ms > 0 ? static_cast<uint64_t>(ms) * 1000000ull : 4000000000ull;
    }();
    return v;
}

// Set-up of the current device, once: sm_103 check, SM count, the status word's
// device address, a stream-ordered memory pool that keeps its memory, kernel
// attributes, and the driver's tensor-map encoder.
int device_state(DeviceState **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(TIM_ERR_UNSUPPORTED_DEVICE, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &d = g_dev[dev];
    if (d.ready) {
        *out = &d;
        return TIM_OK;
    }
    if (d.status_code != TIM_OK)
        return fail(d.status_code, "device %d is not usable by this library", dev);
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3) {
        d.status_code = TIM_ERR_UNSUPPORTED_DEVICE;
        return fail(TIM_ERR_UNSUPPORTED_DEVICE,
                    "device %d is sm_%d%d; this library is built for sm_103a (GB300) only", dev, major, minor);
    }
    if ((e = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_status)) != cudaSuccess)
        return cuda_fail(e, "cudaGetSymbolAddress(status)");
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof props);
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    if ((e = cudaMemPoolCreate(&d.pool, &props)) != cudaSuccess)
        return cuda_fail(e, "cudaMemPoolCreate");
    uint64_t keep = ~0ull;
    if ((e = cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess)
        return cuda_fail(e, "cudaMemPoolSetAttribute");
    if ((e = tim::k1_prepare_device()) != cudaSuccess || (e = tim::k2_prepare_device()) != cudaSuccess ||
        (e = tim::monitor_prepare_device()) != cudaSuccess || (e = tim::gemm_prepare_device()) != cudaSuccess)
        return cuda_fail(e, "cudaFuncSetAttribute");
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
            return fail(TIM_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.ready = true;
    *out = &d;
    return TIM_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// 2-D bf16 tensor map over a row-major [rows, cols] matrix whose rows are
// `row_bytes` apart (a multiple of 16), with a box of [box_rows, 64] and
// 128-byte swizzling; out-of-range elements read as zero.
int encode_bf16_strided(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int64_t row_bytes,
                        uint32_t box_rows)
{
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(tim::K1_BK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(TIM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return TIM_OK;
}

int encode_bf16(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, uint32_t box_rows)
{
    return encode_bf16_strided(m, base, rows, cols, cols * 2, box_rows);
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bytes of the padded copy of a batch's last m-tile (K1_BM rows of h).
size_t tail_pad_bytes(int64_t N, int64_t D)
{
    return tim::k1_needs_tail_pad(N) ? round_up(static_cast<size_t>(tim::K1_BM) * D * 2, 256) : 0;
}

// When N is not a multiple of 16 rows, copies the last m-tile's rows of h into
// `pad` (K1_BM rows, zero past N), maps it in *th_tail and names the m-tile in
// *tail_mt (else *tail_mt = -1 and *th_tail = th).  The kernel reads the same
// values either way: past N both give zeros.
int tail_map(const void *h, int64_t N, int64_t D, void *pad, const CUtensorMap &th, cudaStream_t s,
             CUtensorMap *th_tail, int32_t *tail_mt)
{
    *th_tail = th;
    *tail_mt = -1;
    if (!tim::k1_needs_tail_pad(N))
        return TIM_OK;
    const int64_t m_tiles = (N + tim::K1_BM - 1) / tim::K1_BM;
    const int64_t r0 = (m_tiles - 1) * tim::K1_BM, rows = N - r0;
    const size_t row_bytes = static_cast<size_t>(D) * 2;
    const cudaError_t e = tim::k1_launch_pad_tail(static_cast<const char *>(h) + r0 * row_bytes, rows, D, pad, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "tail pad copy");
    const int rc = encode_bf16(th_tail, pad, tim::K1_BM, D, tim::K1_BM);
    if (rc != TIM_OK)
        return rc;
    *tail_mt = static_cast<int32_t>(m_tiles - 1);
    return TIM_OK;
}

// Rows of one backward chunk: the bf16 logit gradient of a chunk is rows x V
// (5 GB at V = 151936); dh and dW are then two GEMMs per chunk.
constexpr int64_t kBackwardRows = 16384;

// Largest float <= v, and smallest float >= v: a float x then satisfies
// x > float_down(v) <=> x > v, and x < float_up(v) <=> x < v.
float float_down(double v)
{
    float f = static_cast<float>(v);
    if (static_cast<double>(f) > v)
        f = std::nextafter(f, -INFINITY);
    return f;
}

float float_up(double v)
{
    float f = static_cast<float>(v);
    if (static_cast<double>(f) < v)
        f = std::nextafter(f, INFINITY);
    return f;
}

} // namespace

namespace tim {

// Device address of the library's status word on the current device.
cudaError_t status_word_address(int **out)
{
    return cudaGetSymbolAddress(reinterpret_cast<void **>(out), g_status);
}

// Records a message for tim_last_error() on the calling thread; returns code.
int record_error(int code, const char *msg)
{
    if (code == TIM_OK) {
        g_msg[0] = 0;
        return code;
    }
    return fail(code, "%s", msg);
}

} // namespace tim

extern "C" {

int tim_version(void) { return kVersion; }

const char *tim_last_error(void) { return g_msg; }

} // extern "C"

namespace {

// The fused token logprob at 1 / temperature `inv_temp` (every entry point).
// w_segments 1: W bf16 [V, D]; 3: fp32 weights split into three bf16 parts
// [V][3][Dp] (tim_split_weight_fp32).
int token_logprob(const void *h, const void *W, const int32_t *targets, int64_t N, int64_t D, int64_t V,
                  float inv_temp, float *out_logp, float *out_lse, tim_stream_t stream, int w_segments = 1)
{
    if (N < 0 || N >= (int64_t(1) << 31))
        return fail(TIM_ERR_INVALID_ARG, "N = %lld out of range [0, 2^31)", static_cast<long long>(N));
    if (D <= 0 || D % 8 != 0 || D > 65536)
        return fail(TIM_ERR_INVALID_ARG, "D = %lld must be positive, a multiple of 8 and <= 65536",
                    static_cast<long long>(D));
    if (V <= 0 || V >= (int64_t(1) << 31))
        return fail(TIM_ERR_INVALID_ARG, "V = %lld out of range (0, 2^31)", static_cast<long long>(V));
    if (N == 0) {
        g_msg[0] = 0;
        return TIM_OK;
    }
    if (!h || !W || !targets || !out_logp || !out_lse)
        return fail(TIM_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(h, 16) || !aligned(W, 16))
        return fail(TIM_ERR_INVALID_ARG, "h and W must be 16-byte aligned");
    if (!aligned(targets, 4) || !aligned(out_logp, 4) || !aligned(out_lse, 4))
        return fail(TIM_ERR_INVALID_ARG, "targets / outputs must be 4-byte aligned");
    const int64_t m_tiles = (N + tim::K1_BM - 1) / tim::K1_BM;
    const int64_t chunks = tim::k1_num_chunks(V);
    if (m_tiles * chunks >= (int64_t(1) << 31))
        return fail(TIM_ERR_INVALID_ARG, "N x V too large for one call");

    DeviceState *dev = nullptr;
    int rc = device_state(&dev);
    if (rc != TIM_OK)
        return rc;
    CUtensorMap th, tw;
    if ((rc = encode_bf16(&th, h, N, D, tim::K1_BM)) != TIM_OK)
        return rc;
    const int64_t w_cols = w_segments == 1 ? D : 3 * tim::k1_split_cols(D);
    if ((rc = encode_bf16(&tw, W, V, w_cols, tim::K1_W_BOX_ROWS)) != TIM_OK)
        return rc;

    const size_t part_bytes = round_up(static_cast<size_t>(chunks) * N * sizeof(float2), 256);
    const size_t za_bytes = round_up(static_cast<size_t>(N) * sizeof(float), 256);
    const size_t pad_bytes = tail_pad_bytes(N, D);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void *ws = nullptr;
    cudaError_t e =
        cudaMallocFromPoolAsync(&ws, part_bytes + za_bytes + pad_bytes + tim::K1_SCHED_BYTES, dev->pool, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMallocFromPoolAsync(token_logprob workspace)");
    CUtensorMap th_tail;
    int32_t tail_mt = -1;
    if ((rc = tail_map(h, N, D, static_cast<char *>(ws) + part_bytes + za_bytes, th, s, &th_tail, &tail_mt)) !=
        TIM_OK) {
        cudaFreeAsync(ws, s);
        return rc;
    }

    tim::K1Args a{};
    a.targets = targets;
    a.part = static_cast<float2 *>(ws);
    a.za = reinterpret_cast<float *>(static_cast<char *>(ws) + part_bytes);
    a.sched = reinterpret_cast<int *>(static_cast<char *>(ws) + part_bytes + za_bytes + pad_bytes);
    a.status = dev->status;
    a.inv_temp = inv_temp;
    a.N = static_cast<int32_t>(N);
    a.D = static_cast<int32_t>(D);
    a.V = static_cast<int32_t>(V);
    a.w_segments = w_segments;
    a.num_m_tiles = static_cast<int32_t>(m_tiles);
    a.num_chunks = static_cast<int32_t>(chunks);
    tim::k1_set_units(a, m_tiles, chunks, D);
    a.wait_budget_ns = wait_budget_ns();
    a.tail_mt = tail_mt;
    e = tim::k1_launch_main(th, tw, th_tail, a, s);
    if (e == cudaSuccess)
        e = tim::k1_launch_combine(a.part, a.za, targets, a.N, a.V, a.num_chunks, a.inv_temp, out_logp, out_lse,
                                   a.status, s);
    const cudaError_t ef = cudaFreeAsync(ws, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "token_logprob launch");
    if (ef != cudaSuccess)
        return cuda_fail(ef, "cudaFreeAsync(token_logprob workspace)");
    g_msg[0] = 0;
    return TIM_OK;
}

} // namespace

extern "C" {

int tim_token_logprob(const void *h, const void *W, const int32_t *targets, int64_t N, int64_t D,
                      int64_t V, float *out_logp, float *out_lse, tim_stream_t stream)
{
    return token_logprob(h, W, targets, N, D, V, 1.f, out_logp, out_lse, stream);
}

int tim_token_logprob_temperature(const void *h, const void *W, const int32_t *targets, int64_t N, int64_t D,
                                  int64_t V, float temperature, float *out_logp, float *out_lse,
                                  tim_stream_t stream)
{
    if (!(temperature > 0.f) || !std::isfinite(temperature) || !std::isfinite(1.f / temperature))
        return fail(TIM_ERR_INVALID_ARG, "temperature must be positive and finite");
    return token_logprob(h, W, targets, N, D, V, 1.f / temperature, out_logp, out_lse, stream);
}

int tim_mismatch_stats(const float *logp_train, const float *logp_rollout, const uint8_t *mask,
                       const int32_t *seq_offsets, float C, const tim_mismatch_out *out,
                       tim_stream_t stream)
{
    if (!out)
        return fail(TIM_ERR_INVALID_ARG, "out is null");
    const int32_t S = out->num_seqs;
    const int64_t N = out->num_tokens;
    if (S < 0 || N < 0)
        return fail(TIM_ERR_INVALID_ARG, "num_seqs / num_tokens must be >= 0");
    if (S == 0 && N != 0)
        return fail(TIM_ERR_INVALID_ARG, "num_tokens must be 0 when num_seqs is 0");
    if (!(C > 0.f) || !std::isfinite(C))
        return fail(TIM_ERR_INVALID_ARG, "C must be positive and finite");
    const int32_t est = out->seq_estimator == 0 ? 3 : out->seq_estimator;
    if (est != 1 && est != 3)
        return fail(TIM_ERR_INVALID_ARG, "seq_estimator must be 1 or 3");
    if (!seq_offsets || !out->batch_stats)
        return fail(TIM_ERR_INVALID_ARG, "seq_offsets and batch_stats are required");
    if (S > 0 && (!out->seq_stats || !out->seq_flags))
        return fail(TIM_ERR_INVALID_ARG, "seq_stats and seq_flags are required when num_seqs > 0");
    if (N > 0 && (!logp_train || !logp_rollout || !mask))
        return fail(TIM_ERR_INVALID_ARG, "null token array");
    if (!aligned(logp_train, 16) || !aligned(logp_rollout, 16) || !aligned(mask, 16))
        return fail(TIM_ERR_INVALID_ARG, "logp_train, logp_rollout and mask must be 16-byte aligned");
    if (!aligned(seq_offsets, 4) ||
        !aligned(out->seq_stats, 4) || !aligned(out->seq_flags, 4) || !aligned(out->token_weight, 4) ||
        !aligned(out->batch_stats, 8) || !aligned(out->seq_records, 16))
        return fail(TIM_ERR_INVALID_ARG, "misaligned array");

    DeviceState *dev = nullptr;
    int rc = device_state(&dev);
    if (rc != TIM_OK)
        return rc;

    const double lc = std::log(static_cast<double>(C));
    const float lcd = float_down(lc);
    const float tau = std::isnan(out->tau_seq) ? static_cast<float>((static_cast<double>(C) - 1.0) - lc)
                                               : out->tau_seq;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void *ws = nullptr;
    const size_t rec_bytes = S > 0 ? tim::k2_workspace_bytes(S) : 0;
    if (rec_bytes > 0) {
        cudaError_t e = cudaMallocFromPoolAsync(&ws, rec_bytes, dev->pool, s);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMallocFromPoolAsync(mismatch workspace)");
    }
    tim::K2Args a;
    a.l_tr = logp_train;
    a.l_ro = logp_rollout;
    a.mask = mask;
    a.off = seq_offsets;
    a.S = S;
    a.N = N;
    a.C = C;
    a.log_c_down = lcd;
    a.tau = tau;
    a.wait_budget_ns = wait_budget_ns();
    a.estimator = est;
    a.token_weight = out->token_weight;
    a.seq_stats = out->seq_stats;
    a.seq_flags = out->seq_flags;
    a.batch = out->batch_stats;
    a.claim = static_cast<int *>(ws);
    a.blk_done = a.claim ? a.claim + 1 : nullptr;
    uint32_t *const ws_rec = S > 0 ? reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + 256) : nullptr;
    a.rec = out->seq_records ? out->seq_records : ws_rec;
    a.part = S > 0 ? ws_rec + static_cast<size_t>(S) * tim::K2_REC_WORDS : nullptr;
    a.stats_vec = aligned(out->seq_stats, 16) ? 1 : 0;
    a.status = dev->status;
    cudaError_t e = tim::k2_launch(a, dev->sms, s);
    cudaError_t ef = ws ? cudaFreeAsync(ws, s) : cudaSuccess;
    if (e != cudaSuccess)
        return cuda_fail(e, "mismatch_stats launch");
    if (ef != cudaSuccess)
        return cuda_fail(ef, "cudaFreeAsync(mismatch workspace)");
    g_msg[0] = 0;
    return TIM_OK;
}

int tim_token_logprob_backward(const void *h, const void *W, const int32_t *targets, const float *grad_logp,
                               const float *lse, int64_t N, int64_t D, int64_t V, float temperature, float *dh,
                               float *dW, int accumulate_dW, tim_stream_t stream)
{
    if (N < 0 || N >= (int64_t(1) << 31))
        return fail(TIM_ERR_INVALID_ARG, "N = %lld out of range [0, 2^31)", static_cast<long long>(N));
    if (D <= 0 || D % 8 != 0 || D > 65536)
        return fail(TIM_ERR_INVALID_ARG, "D = %lld must be positive, a multiple of 8 and <= 65536",
                    static_cast<long long>(D));
    if (V <= 0 || V >= (int64_t(1) << 31))
        return fail(TIM_ERR_INVALID_ARG, "V = %lld out of range (0, 2^31)", static_cast<long long>(V));
    if (!(temperature > 0.f) || !std::isfinite(temperature) || !std::isfinite(1.f / temperature))
        return fail(TIM_ERR_INVALID_ARG, "temperature must be positive and finite");
    if (!W || !dW)
        return fail(TIM_ERR_INVALID_ARG, "W and dW are required");
    if (N > 0 && (!h || !targets || !grad_logp || !lse || !dh))
        return fail(TIM_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(h, 16) || !aligned(W, 16) || !aligned(dh, 16) || !aligned(dW, 16))
        return fail(TIM_ERR_INVALID_ARG, "h, W, dh and dW must be 16-byte aligned");
    if (!aligned(targets, 4) || !aligned(grad_logp, 4) || !aligned(lse, 4))
        return fail(TIM_ERR_INVALID_ARG, "targets / grad_logp / lse must be 4-byte aligned");

    DeviceState *dev = nullptr;
    int rc = device_state(&dev);
    if (rc != TIM_OK)
        return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (N == 0) {   // no rows: dW = 0 unless accumulating
        if (!accumulate_dW) {
            const cudaError_t e = cudaMemsetAsync(dW, 0, static_cast<size_t>(V) * D * sizeof(float), s);
            if (e != cudaSuccess)
                return cuda_fail(e, "cudaMemsetAsync(dW)");
        }
        g_msg[0] = 0;
        return TIM_OK;
    }
    // rows in chunks of at most kBackwardRows: dz of one chunk, bf16 [rows][Vp]
    const int64_t Vp = (V + 7) / 8 * 8;
    const int64_t rows_max = std::min<int64_t>(kBackwardRows, (N + 255) / 256 * 256);
    const size_t dz_bytes = round_up(static_cast<size_t>(rows_max) * Vp * 2, 256);
    const size_t pad_bytes = round_up(static_cast<size_t>(tim::K1_BM) * D * 2, 256);
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, dz_bytes + pad_bytes + tim::K1_SCHED_BYTES, dev->pool, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMallocFromPoolAsync(backward workspace)");
    int *sched = reinterpret_cast<int *>(static_cast<char *>(ws) + dz_bytes + pad_bytes);
    CUtensorMap tw, tw_mn;
    if ((rc = encode_bf16(&tw, W, V, D, tim::K1_W_BOX_ROWS)) != TIM_OK ||
        (rc = encode_bf16(&tw_mn, W, V, D, tim::G_MNMAJOR_BOX_ROWS)) != TIM_OK) {
        cudaFreeAsync(ws, s);
        return rc;
    }
    const int64_t chunks_v = tim::k1_num_chunks(V);
    const int32_t n_blocks = static_cast<int32_t>((D + tim::G_BN - 1) / tim::G_BN);
    for (int64_t r0 = 0; r0 < N && rc == TIM_OK; r0 += rows_max) {
        const int64_t n = std::min<int64_t>(rows_max, N - r0);
        const void *hc = static_cast<const uint16_t *>(h) + r0 * D;
        CUtensorMap th, th_tail, th_mn, tdz_k, tdz_mn;
        int32_t tail_mt = -1;
        // dz is read up to column V only (the row padding past V holds no data
        // and reads as zero), its rows Vp apart
        if ((rc = encode_bf16(&th, hc, n, D, tim::K1_BM)) != TIM_OK ||
            (rc = tail_map(hc, n, D, static_cast<char *>(ws) + dz_bytes, th, s, &th_tail, &tail_mt)) != TIM_OK ||
            (rc = encode_bf16(&th_mn, hc, n, D, tim::G_MNMAJOR_BOX_ROWS)) != TIM_OK ||
            (rc = encode_bf16_strided(&tdz_k, ws, n, V, Vp * 2, tim::G_KMAJOR_BOX_ROWS)) != TIM_OK ||
            (rc = encode_bf16_strided(&tdz_mn, ws, n, V, Vp * 2, tim::G_MNMAJOR_BOX_ROWS)) != TIM_OK)
            break;
        const int64_t m_tiles = (n + tim::K1_BM - 1) / tim::K1_BM;
        tim::K1Args a{};
        a.targets = targets + r0;
        a.sched = sched;
        a.status = dev->status;
        a.inv_temp = 1.f / temperature;
        a.N = static_cast<int32_t>(n);
        a.D = static_cast<int32_t>(D);
        a.V = static_cast<int32_t>(V);
        a.w_segments = 1;
        a.num_m_tiles = static_cast<int32_t>(m_tiles);
        a.num_chunks = static_cast<int32_t>(chunks_v);
        tim::k1_set_units(a, m_tiles, chunks_v, D);
        a.wait_budget_ns = wait_budget_ns();
        a.grad = grad_logp + r0;
        a.lse_in = lse + r0;
        a.dz = static_cast<uint16_t *>(ws);
        a.dz_ld = Vp;
        a.tail_mt = tail_mt;
        if ((e = tim::k1_launch_main(th, tw, th_tail, a, s, 1)) != cudaSuccess) {
            rc = cuda_fail(e, "backward dz launch");
            break;
        }
        // one launch, two GEMMs (dh's tiles claimed first, then dW's):
        // dh rows of the chunk = dz W: A = dz [n][V] K-major, B = W [V][D] MN-major, K = V;
        // dW (+)= dz^T h: A = dz^T (dz [n][V] read MN-major), B = h [n][D] MN-major,
        // K = n; chunks in row order, each adding to the sum of the chunks before
        tim::GemmArgs g{};
        tim::GemmProblem &ph = g.p[0], &pw = g.p[1];
        ph.C = dh + r0 * D;
        ph.ldc = D;
        ph.M = static_cast<int32_t>(n);
        ph.N = static_cast<int32_t>(D);
        ph.K = static_cast<int32_t>(V);
        ph.n_blocks = n_blocks;
        ph.units = static_cast<int32_t>((n + 2 * tim::G_BM - 1) / (2 * tim::G_BM)) * n_blocks;
        ph.accumulate = 0;
        ph.b_keep = 0;
        pw = ph;
        pw.C = dW;
        pw.M = static_cast<int32_t>(V);
        pw.K = static_cast<int32_t>(n);
        pw.units = static_cast<int32_t>((V + 2 * tim::G_BM - 1) / (2 * tim::G_BM)) * n_blocks;
        pw.accumulate = (r0 > 0 || accumulate_dW) ? 1 : 0;
        pw.b_keep = 1;   // h of the chunk (at most 16384 x D bf16) is read by every dW tile
        g.sched = sched;
        g.status = dev->status;
        g.wait_budget_ns = wait_budget_ns();
        const CUtensorMap maps_a[2] = {tdz_k, tdz_mn}, maps_b[2] = {tw_mn, th_mn};
        if ((e = tim::gemm_launch(maps_a, maps_b, g, s)) != cudaSuccess) {
            rc = cuda_fail(e, "backward dh / dW launch");
            break;
        }
    }
    const cudaError_t ef = cudaFreeAsync(ws, s);
    if (rc != TIM_OK)
        return rc;
    if (ef != cudaSuccess)
        return cuda_fail(ef, "cudaFreeAsync(backward workspace)");
    g_msg[0] = 0;
    return TIM_OK;
}

int64_t tim_split_weight_bytes(int64_t V, int64_t D)
{
    if (V <= 0 || D <= 0 || V >= (int64_t(1) << 31) || D > 65536)
        return -1;
    return V * 3 * tim::k1_split_cols(D) * 2;
}

int tim_split_weight_fp32(const float *W, int64_t V, int64_t D, void *W_split, tim_stream_t stream)
{
    if (V <= 0 || V >= (int64_t(1) << 31) || D <= 0 || D % 8 != 0 || D > 65536)
        return fail(TIM_ERR_INVALID_ARG, "V must be in (0, 2^31), D positive, a multiple of 8 and <= 65536");
    if (!W || !W_split)
        return fail(TIM_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(W, 16) || !aligned(W_split, 16))
        return fail(TIM_ERR_INVALID_ARG, "W and W_split must be 16-byte aligned");
    DeviceState *dev = nullptr;
    int rc = device_state(&dev);
    if (rc != TIM_OK)
        return rc;
    const cudaError_t e = tim::k1_launch_split(W, V, D, W_split, dev->sms, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "split_weight_fp32 launch");
    g_msg[0] = 0;
    return TIM_OK;
}

int tim_token_logprob_fp32_head(const void *h, const void *W_split, const int32_t *targets, int64_t N, int64_t D,
                                int64_t V, float temperature, float *out_logp, float *out_lse, tim_stream_t stream)
{
    if (!(temperature > 0.f) || !std::isfinite(temperature) || !std::isfinite(1.f / temperature))
        return fail(TIM_ERR_INVALID_ARG, "temperature must be positive and finite");
    return token_logprob(h, W_split, targets, N, D, V, 1.f / temperature, out_logp, out_lse, stream, 3);
}

int tim_mismatch_fold(const uint32_t *seq_records, int32_t num_seqs, double *batch_stats, tim_stream_t stream)
{
    const int32_t S = num_seqs;
    if (S < 0)
        return fail(TIM_ERR_INVALID_ARG, "num_seqs must be >= 0");
    if (!batch_stats || (S > 0 && !seq_records))
        return fail(TIM_ERR_INVALID_ARG, "seq_records and batch_stats are required");
    if (!aligned(seq_records, 16) || !aligned(batch_stats, 8))
        return fail(TIM_ERR_INVALID_ARG, "misaligned array");
    DeviceState *dev = nullptr;
    int rc = device_state(&dev);
    if (rc != TIM_OK)
        return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void *ws = nullptr;
    if (S > 0) {
        const cudaError_t e = cudaMallocFromPoolAsync(&ws, tim::k2_fold_workspace_bytes(S), dev->pool, s);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMallocFromPoolAsync(fold workspace)");
    }
    tim::K2Args a{};
    a.S = S;
    a.batch = batch_stats;
    a.claim = static_cast<int *>(ws);
    a.blk_done = a.claim ? a.claim + 1 : nullptr;
    a.rec = const_cast<uint32_t *>(seq_records);   // read only by the fold
    a.part = S > 0 ? reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + 256) : nullptr;
    a.status = dev->status;
    const cudaError_t e = tim::k2_launch_fold(a, s);
    const cudaError_t ef = ws ? cudaFreeAsync(ws, s) : cudaSuccess;
    if (e != cudaSuccess)
        return cuda_fail(e, "mismatch_fold launch");
    if (ef != cudaSuccess)
        return cuda_fail(ef, "cudaFreeAsync(fold workspace)");
    g_msg[0] = 0;
    return TIM_OK;
}

int tim_mismatch_monitor(const float *logp_train, const float *logp_rollout, const uint8_t *mask, int64_t N,
                         float tau_tok, uint8_t *token_reject, double *out, tim_stream_t stream)
{
    if (N < 0 || N >= (int64_t(1) << 31))
        return fail(TIM_ERR_INVALID_ARG, "N must be in [0, 2^31)");
    if (!(tau_tok >= 0.f) || !std::isfinite(tau_tok))
        return fail(TIM_ERR_INVALID_ARG, "tau_tok must be >= 0 and finite");
    if (!out)
        return fail(TIM_ERR_INVALID_ARG, "out is required");
    if (N > 0 && (!logp_train || !logp_rollout || !mask))
        return fail(TIM_ERR_INVALID_ARG, "null token array");
    if (!aligned(logp_train, 16) || !aligned(logp_rollout, 16) || !aligned(mask, 16) || !aligned(token_reject, 16))
        return fail(TIM_ERR_INVALID_ARG, "logp_train, logp_rollout, mask and token_reject must be 16-byte aligned");
    if (!aligned(out, 8))
        return fail(TIM_ERR_INVALID_ARG, "misaligned array");

    DeviceState *dev = nullptr;
    int rc = device_state(&dev);
    if (rc != TIM_OK)
        return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, tim::monitor_workspace_bytes(N), dev->pool, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMallocFromPoolAsync(monitor workspace)");
    tim::MonArgs a;
    a.l_tr = logp_train;
    a.l_ro = logp_rollout;
    a.mask = mask;
    a.N = N;
    a.tau_tok = tau_tok;
    a.reject = token_reject;
    a.out = out;
    tim::monitor_bind(a, ws, N);
    a.status = dev->status;
    a.wait_budget_ns = wait_budget_ns();
    e = tim::monitor_launch(a, dev->sms, s);
    cudaError_t ef = cudaFreeAsync(ws, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "mismatch_monitor launch");
    if (ef != cudaSuccess)
        return cuda_fail(ef, "cudaFreeAsync(monitor workspace)");
    g_msg[0] = 0;
    return TIM_OK;
}

int tim_tis_ppo(const float *logp_theta, const float *logp_old, const float *logp_rollout, const float *advantages,
                const uint8_t *mask, const int32_t *seq_offsets, float eps_low, float eps_high, float C,
                const tim_ppo_out *out, tim_stream_t stream)
{
    if (!out)
        return fail(TIM_ERR_INVALID_ARG, "out is null");
    const int32_t S = out->num_seqs;
    const int64_t N = out->num_tokens;
    if (S < 0 || N < 0)
        return fail(TIM_ERR_INVALID_ARG, "num_seqs / num_tokens must be >= 0");
    if (S == 0 && N != 0)
        return fail(TIM_ERR_INVALID_ARG, "num_tokens must be 0 when num_seqs is 0");
    if (!(C > 0.f) || !std::isfinite(C))
        return fail(TIM_ERR_INVALID_ARG, "C must be positive and finite");
    if (!(eps_low >= 0.f && eps_low < 1.f))
        return fail(TIM_ERR_INVALID_ARG, "eps_low must be in [0, 1)");
    if (!(eps_high >= 0.f) || !std::isfinite(eps_high))
        return fail(TIM_ERR_INVALID_ARG, "eps_high must be >= 0 and finite");
    if (!seq_offsets || !out->batch_stats)
        return fail(TIM_ERR_INVALID_ARG, "seq_offsets and batch_stats are required");
    if (S > 0 && !out->seq_loss)
        return fail(TIM_ERR_INVALID_ARG, "seq_loss is required when num_seqs > 0");
    if (N > 0 && (!logp_theta || !logp_old || !logp_rollout || !advantages || !mask))
        return fail(TIM_ERR_INVALID_ARG, "null token array");
    if (!aligned(logp_theta, 4) || !aligned(logp_old, 4) || !aligned(logp_rollout, 4) || !aligned(advantages, 4) ||
        !aligned(seq_offsets, 4) || !aligned(out->token_loss, 4) || !aligned(out->token_grad, 4) ||
        !aligned(out->seq_loss, 4) || !aligned(out->batch_stats, 8))
        return fail(TIM_ERR_INVALID_ARG, "misaligned array");

    DeviceState *dev = nullptr;
    int rc = device_state(&dev);
    if (rc != TIM_OK)
        return rc;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void *ws = nullptr;
    if (S > 0) {
        cudaError_t e = cudaMallocFromPoolAsync(&ws, tim::ppo_workspace_bytes(S), dev->pool, s);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMallocFromPoolAsync(ppo workspace)");
    }
    tim::PpoArgs a;
    a.l_th = logp_theta;
    a.l_old = logp_old;
    a.l_ro = logp_rollout;
    a.adv = advantages;
    a.mask = mask;
    a.off = seq_offsets;
    a.S = S;
    a.N = N;
    a.C = C;
    a.log_c_down = float_down(std::log(static_cast<double>(C)));
    a.log_hi_down = float_down(std::log1p(static_cast<double>(eps_high)));
    a.log_lo_up = float_up(std::log1p(-static_cast<double>(eps_low)));
    a.r_hi = static_cast<float>(1.0 + static_cast<double>(eps_high));
    a.r_lo = static_cast<float>(1.0 - static_cast<double>(eps_low));
    a.token_loss = out->token_loss;
    a.token_grad = out->token_grad;
    a.seq_loss = out->seq_loss;
    a.batch = out->batch_stats;
    a.rec = static_cast<uint32_t *>(ws);
    a.part = S > 0 ? a.rec + round_up(static_cast<size_t>(S) * tim::PPO_REC_WORDS, 64) : nullptr;
    a.ticket = S > 0 ? a.part + round_up(static_cast<size_t>((S + tim::PPO_FOLD_SEQS - 1) / tim::PPO_FOLD_SEQS) *
                                             tim::PPO_PART_WORDS, 64)
                     : nullptr;
    a.claim = S > 0 ? reinterpret_cast<int *>(a.ticket + 32) : nullptr;   // its own 128-byte line
    a.status = dev->status;
    cudaError_t e = tim::ppo_launch(a, dev->sms, s);
    cudaError_t ef = ws ? cudaFreeAsync(ws, s) : cudaSuccess;
    if (e != cudaSuccess)
        return cuda_fail(e, "tis_ppo launch");
    if (ef != cudaSuccess)
        return cuda_fail(ef, "cudaFreeAsync(ppo workspace)");
    g_msg[0] = 0;
    return TIM_OK;
}

int tim_check(tim_stream_t stream)
{
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaStreamSynchronize");
    DeviceState *dev = nullptr;
    int rc = device_state(&dev);
    if (rc != TIM_OK)
        return rc;
    int v = 0;
    if ((e = cudaMemcpyAsync(&v, dev->status, sizeof v, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return cuda_fail(e, "read status");
    if ((e = cudaMemsetAsync(dev->status, 0, sizeof v, s)) != cudaSuccess)
        return cuda_fail(e, "clear status");
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess)
        return cuda_fail(e, "cudaStreamSynchronize");
    if (v != TIM_OK)
        return fail(v, "a kernel recorded status %d (%s)", v,
                    v == TIM_ERR_TIMEOUT ? "pipeline wait ran out of time" : "bad input data");
    g_msg[0] = 0;
    return TIM_OK;
}

int tim_debug_violation(int64_t out[4], tim_stream_t stream)
{
    if (!out)
        return fail(TIM_ERR_INVALID_ARG, "out is null");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    DeviceState *dev = nullptr;
    int rc = device_state(&dev);
    if (rc != TIM_OK)
        return rc;
    int w[tim::STATUS_WORDS] = {};
    cudaError_t e = cudaStreamSynchronize(s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(w, dev->status, sizeof w, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)   // words 1..7: the record (the status itself is tim_check's)
        e = cudaMemsetAsync(dev->status + 1, 0, sizeof w - sizeof(int), s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(e, "read the violation record");
    long long index = 0;
    unsigned long long value = 0;
    std::memcpy(&index, w + 2, sizeof index);
    std::memcpy(&value, w + 4, sizeof value);
    out[0] = w[1];
    out[1] = index;
    out[2] = static_cast<int64_t>(value);
    out[3] = 0;
    g_msg[0] = 0;
    return TIM_OK;
}

int tim_debug_build(void)
{
#ifdef TIM_DEBUG
    return 1;
#else
    return 0;
#endif
}

} // extern "C"
