// api.cu -- the extern "C" boundary declared in include/mxfp8.h.
//
// Host-side validation happens before any launch; every entry point is
// asynchronous on the caller's stream and never allocates.  The layer's
// steps follow vLLM PR #52204 "[Kernel] Add FlashInfer TRTLLM MXFP8 linear
// backend": process_weights_after_loading -> mxfp8_prepare_weight,
// flashinfer_mxfp8_quantize_8x4 -> mxfp8_quantize_act, mm_mxfp8 + slice +
// bias -> mxfp8_gemm, apply_weights -> mxfp8_linear.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include <algorithm>
#include <atomic>
#include <vector>

#include "../../include/mxfp8.h"
#include "../../include/mxfp8_moe.h"
#include "../../include/mxfp8_testing.h"
#include "internal.h"

namespace {

thread_local int t_last_cuda_error = 0;
// Testing hooks (mxfp8_set_schedule), read by every call on any thread.
std::atomic<int> g_force_tt{0};
std::atomic<int> g_force_split{0};
std::atomic<int> g_force_fuse{-1};

// Per-device capability cache, filled by whichever thread calls first.
struct DeviceInfo {
    std::atomic<int> checked;  // 0 unknown, 1 supported, -1 unsupported
    std::atomic<int> sms;
};
DeviceInfo g_dev[64];  // static storage: starts zeroed

mxfp8_status cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return MXFP8_ERR_CUDA;
}

}  // namespace

// The code mxfp8_last_cuda_error() reports on this thread (other entry
// points of the library record their failed CUDA calls here too).
void mxk::record_cuda_error(int e) { t_last_cuda_error = e; }

namespace {

// Current device must be compute capability 10.3 (GB300).
mxfp8_status device_sms(int* sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= 64) return MXFP8_ERR_UNSUPPORTED_DEVICE;
    DeviceInfo& d = g_dev[dev];
    int checked = d.checked.load(std::memory_order_acquire);
    if (checked == 0) {  // racing first calls write the same values
        int major = 0, minor = 0, count = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e);
        d.sms.store(count, std::memory_order_relaxed);
        checked = (major == 10 && minor == 3) ? 1 : -1;
        d.checked.store(checked, std::memory_order_release);
    }
    if (checked < 0) return MXFP8_ERR_UNSUPPORTED_DEVICE;
    *sms = d.sms.load(std::memory_order_relaxed);
    return MXFP8_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t ceil_to(int64_t v, int64_t q) { return (v + q - 1) / q * q; }

// Shape limits keep every in-kernel index (int32 token/row counts, int64
// byte offsets) in range.
constexpr int64_t kMaxRows = (int64_t(1) << 31) - 256;
constexpr int64_t kMaxK = int64_t(1) << 20;

mxfp8_status check_weight(const mxfp8_weight* w) {
    if (!w || !w->q || !w->sf) return MXFP8_ERR_INVALID_ARG;
    if (w->num_experts < 1 || w->num_experts > 1024 || w->n < 1 || w->k < 1) return MXFP8_ERR_INVALID_ARG;
    if (w->k % 256 != 0) return MXFP8_ERR_K_NOT_MULTIPLE_OF_256;
    if (w->k > kMaxK || w->n_pad != ceil_to(w->n, 128) || w->num_experts * w->n_pad > kMaxRows)
        return MXFP8_ERR_INVALID_ARG;
    if (!aligned16(w->q) || !aligned16(w->sf)) return MXFP8_ERR_MISALIGNED;
    return MXFP8_OK;
}

}  // namespace

extern "C" {

size_t mxfp8_act_scale_bytes(int64_t m, int64_t k) {
    if (m < 0 || m > kMaxRows || k <= 0 || k > kMaxK || k % 32 != 0) return 0;
    return static_cast<size_t>(ceil_to(m, 8) * ceil_to(k / 32, 4));
}

size_t mxfp8_weight_bytes(int64_t n, int64_t k) {
    if (n <= 0 || n > kMaxRows || k <= 0 || k > kMaxK) return 0;
    return static_cast<size_t>(ceil_to(n, 128) * k);
}

size_t mxfp8_weight_scale_bytes(int64_t n, int64_t k) {
    if (n <= 0 || n > kMaxRows || k <= 0 || k > kMaxK || k % 32 != 0) return 0;
    return static_cast<size_t>(ceil_to(n, 128) * (k / 32));
}

size_t mxfp8_linear_workspace_bytes(int64_t m, int64_t k) {
    if (m < 0 || m > kMaxRows || k <= 0 || k > kMaxK || k % 32 != 0) return 0;
    return static_cast<size_t>(ceil_to(m * k, 256)) + mxfp8_act_scale_bytes(m, k);
}

mxfp8_status mxfp8_weight_view(mxfp8_weight* w, int64_t num_experts, int64_t n, int64_t k, void* q,
                               void* sf) {
    if (!w) return MXFP8_ERR_INVALID_ARG;
    w->num_experts = num_experts;
    w->n = n;
    w->n_pad = n > 0 ? ceil_to(n, 128) : 0;
    w->k = k;
    w->q = q;
    w->sf = sf;
    return check_weight(w);
}

mxfp8_status mxfp8_prepare_weight(const void* src, mxfp8_in_dtype dtype, const mxfp8_weight* w,
                                  void* stream) {
    mxfp8_status st = check_weight(w);
    if (st != MXFP8_OK) return st;
    if (!src || (dtype != MXFP8_IN_F32 && dtype != MXFP8_IN_BF16)) return MXFP8_ERR_INVALID_ARG;
    if (!aligned16(src)) return MXFP8_ERR_MISALIGNED;
    int sms = 0;
    if ((st = device_sms(&sms)) != MXFP8_OK) return st;
    cudaError_t e = mxk::launch_prepare_weight(src, dtype == MXFP8_IN_BF16, w->num_experts, w->n, w->n_pad,
                                               w->k, static_cast<uint8_t*>(w->q),
                                               static_cast<uint8_t*>(w->sf), sms,
                                               static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MXFP8_OK : cuda_fail(e);
}

mxfp8_status mxfp8_quantize_act(const void* x, int64_t m, int64_t k, void* q, void* sf, void* stream) {
    if (m < 0 || k < 1) return MXFP8_ERR_INVALID_ARG;
    if (k % 256 != 0) return MXFP8_ERR_K_NOT_MULTIPLE_OF_256;
    if (m > kMaxRows || k > kMaxK) return MXFP8_ERR_INVALID_ARG;
    if (m == 0) return MXFP8_OK;
    if (!x || !q || !sf) return MXFP8_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q) || !aligned16(sf)) return MXFP8_ERR_MISALIGNED;
    int sms = 0;
    mxfp8_status st = device_sms(&sms);
    if (st != MXFP8_OK) return st;
    cudaError_t e = mxk::launch_quant_act(x, m, k, static_cast<uint8_t*>(q), static_cast<uint8_t*>(sf),
                                          sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MXFP8_OK : cuda_fail(e);
}

static mxk::GemmProblem make_problem(const void* qa, const void* sfa, int64_t m, const mxfp8_weight* w,
                                     const void* bias, void* y, const int32_t* offsets, const void* x) {
    mxk::GemmProblem p;
    p.qa = static_cast<const uint8_t*>(qa);
    p.sfa = static_cast<const uint8_t*>(sfa);
    p.m = m;
    p.wq = static_cast<const uint8_t*>(w->q);
    p.wsf = static_cast<const uint8_t*>(w->sf);
    p.experts = w->num_experts;
    p.n = w->n;
    p.n_pad = w->n_pad;
    p.k = w->k;
    p.bias = bias;
    p.y = y;
    p.offsets = offsets;
    p.x = x;
    p.gated = false;
    p.sf128 = false;
    p.hq = nullptr;
    p.hsf = nullptr;
    return p;
}

// Set by the autotuner while it times one candidate on this thread.
thread_local const mxk::GemmSchedule* t_override = nullptr;

// Schedule of a call: the autotuner's candidate, else the testing hooks if
// set, else the tactic table, else the built-in heuristic.
static mxk::GemmSchedule select_schedule(const mxk::GemmProblem& p, int sms, int kind) {
    if (t_override) return *t_override;
    const int ftt = g_force_tt.load(std::memory_order_relaxed);
    const int fsplit = g_force_split.load(std::memory_order_relaxed);
    const int ffuse = g_force_fuse.load(std::memory_order_relaxed);
    if (ftt != 0 || fsplit != 0 || ffuse != -1) return mxk::choose_schedule(p, sms, ftt, fsplit, ffuse);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;  // as the table operations
    mxk::GemmSchedule s;
    if (mxk::tactic_lookup(dev, kind, p.m, p.n, p.k, p.experts, &s)) {
        if (s.fuse_quant && p.x == nullptr) s.fuse_quant = false;
        return s;
    }
    return mxk::choose_schedule(p, sms, 0, 0, -1);
}

static mxfp8_status launch_status(cudaError_t e, bool enc_fail) {
    if (enc_fail) return MXFP8_ERR_INVALID_ARG;
    return e == cudaSuccess ? MXFP8_OK : cuda_fail(e);
}

mxfp8_status mxfp8_gemm(const void* qa, const void* sfa, int64_t m, const mxfp8_weight* w,
                        const void* bias, void* y, void* stream) {
    mxfp8_status st = check_weight(w);
    if (st != MXFP8_OK) return st;
    if (w->num_experts != 1 || m < 0 || m > kMaxRows) return MXFP8_ERR_INVALID_ARG;
    if (m == 0) return MXFP8_OK;
    if (!qa || !sfa || !y) return MXFP8_ERR_INVALID_ARG;
    if (!aligned16(qa) || !aligned16(sfa)) return MXFP8_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(y) & 1u) || (reinterpret_cast<uintptr_t>(bias) & 1u))
        return MXFP8_ERR_MISALIGNED;
    int sms = 0;
    if ((st = device_sms(&sms)) != MXFP8_OK) return st;
    const mxk::GemmProblem p = make_problem(qa, sfa, m, w, bias, y, nullptr, nullptr);
    const mxk::GemmSchedule sch = select_schedule(p, sms, mxk::kTacticGemm);
    bool enc_fail = false;
    cudaError_t e = mxk::launch_gemm(p, sch, sms, static_cast<cudaStream_t>(stream), &enc_fail);
    return launch_status(e, enc_fail);
}

static mxfp8_status linear_common(const void* x, int64_t m, const int32_t* offsets,
                                  const mxfp8_weight* w, const void* bias, void* y, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    mxfp8_status st = check_weight(w);
    if (st != MXFP8_OK) return st;
    if (m < 0 || m > kMaxRows) return MXFP8_ERR_INVALID_ARG;
    if (m == 0) return MXFP8_OK;
    if (!x || !y || !workspace) return MXFP8_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(workspace)) return MXFP8_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(y) & 1u) || (reinterpret_cast<uintptr_t>(bias) & 1u))
        return MXFP8_ERR_MISALIGNED;
    if (workspace_bytes < mxfp8_linear_workspace_bytes(m, w->k)) return MXFP8_ERR_WORKSPACE_TOO_SMALL;
    int sms = 0;
    if ((st = device_sms(&sms)) != MXFP8_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* qa = static_cast<uint8_t*>(workspace);
    uint8_t* sfa = qa + ceil_to(m * w->k, 256);
    // Small M: the GEMM quantizes its own K slices of x (no separate launch,
    // the workspace stays unused).  Otherwise quantize into the workspace.
    const mxk::GemmProblem p = make_problem(qa, sfa, m, w, bias, y, offsets, offsets ? nullptr : x);
    const mxk::GemmSchedule sch = select_schedule(p, sms, offsets ? mxk::kTacticGrouped : mxk::kTacticLinear);
    if (!sch.fuse_quant) {
        cudaError_t e = mxk::launch_quant_act(x, m, w->k, qa, sfa, sms, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    bool enc_fail = false;
    cudaError_t e = mxk::launch_gemm(p, sch, sms, s, &enc_fail);
    return launch_status(e, enc_fail);
}

mxfp8_status mxfp8_linear(const void* x, int64_t m, const mxfp8_weight* w, const void* bias, void* y,
                          void* workspace, size_t workspace_bytes, void* stream) {
    if (w && w->num_experts != 1) return MXFP8_ERR_INVALID_ARG;
    return linear_common(x, m, nullptr, w, bias, y, workspace, workspace_bytes, stream);
}

mxfp8_status mxfp8_grouped_linear(const void* x_sorted, int64_t rows, const int32_t* expert_offsets,
                                  const mxfp8_weight* w, const void* bias, void* y, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    if (!expert_offsets) return MXFP8_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(expert_offsets) & 3u)) return MXFP8_ERR_MISALIGNED;
    return linear_common(x_sorted, rows, expert_offsets, w, bias, y, workspace, workspace_bytes, stream);
}

// -------------------------------------------------- host activations/output
size_t mxfp8_linear_host_workspace_bytes(int64_t m, int64_t n, int64_t k) {
    if (m < 0 || m > kMaxRows || n < 1 || n > kMaxRows || k <= 0 || k > kMaxK || k % 32 != 0) return 0;
    return static_cast<size_t>(ceil_to(m * k * 2, 256) + ceil_to(m * n * 2, 256)) +
           mxfp8_linear_workspace_bytes(m, k);
}

mxfp8_status mxfp8_linear_host(const void* x_host, int64_t m, const mxfp8_weight* w, const void* bias,
                               void* y_host, void* workspace, size_t workspace_bytes, void* stream) {
    mxfp8_status st = check_weight(w);
    if (st != MXFP8_OK) return st;
    if (w->num_experts != 1 || m < 0 || m > kMaxRows) return MXFP8_ERR_INVALID_ARG;
    if (m == 0) return MXFP8_OK;
    if (!x_host || !y_host || !workspace) return MXFP8_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return MXFP8_ERR_MISALIGNED;
    if (workspace_bytes < mxfp8_linear_host_workspace_bytes(m, w->n, w->k)) return MXFP8_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* xd = static_cast<uint8_t*>(workspace);
    uint8_t* yd = xd + ceil_to(m * w->k * 2, 256);
    uint8_t* ws = yd + ceil_to(m * w->n * 2, 256);
    const size_t x_bytes = static_cast<size_t>(m * w->k * 2), y_bytes = static_cast<size_t>(m * w->n * 2);
    cudaError_t e = cudaMemcpyAsync(xd, x_host, x_bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e);
    st = linear_common(xd, m, nullptr, w, bias, yd, ws, mxfp8_linear_workspace_bytes(m, w->k), stream);
    if (st != MXFP8_OK) return st;
    e = cudaMemcpyAsync(y_host, yd, y_bytes, cudaMemcpyDeviceToHost, s);
    return e == cudaSuccess ? MXFP8_OK : cuda_fail(e);
}

// -------------------------------------------------- 128x4 activation scales
size_t mxfp8_act_scale_bytes_128x4(int64_t m, int64_t k) {
    if (m < 0 || m > kMaxRows || k <= 0 || k > kMaxK || k % 128 != 0) return 0;
    return static_cast<size_t>(ceil_to(m, 128) * (k / 32));
}

size_t mxfp8_linear_128x4_workspace_bytes(int64_t m, int64_t k) {
    if (m < 0 || m > kMaxRows || k <= 0 || k > kMaxK || k % 128 != 0) return 0;
    return static_cast<size_t>(ceil_to(m * k, 256)) + mxfp8_act_scale_bytes_128x4(m, k);
}

mxfp8_status mxfp8_quantize_act_128x4(const void* x, int64_t m, int64_t k, void* q, void* sf, void* stream) {
    if (m < 0 || k < 1) return MXFP8_ERR_INVALID_ARG;
    if (k % 256 != 0) return MXFP8_ERR_K_NOT_MULTIPLE_OF_256;
    if (m > kMaxRows || k > kMaxK) return MXFP8_ERR_INVALID_ARG;
    if (m == 0) return MXFP8_OK;
    if (!x || !q || !sf) return MXFP8_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q) || !aligned16(sf)) return MXFP8_ERR_MISALIGNED;
    int sms = 0;
    mxfp8_status st = device_sms(&sms);
    if (st != MXFP8_OK) return st;
    cudaError_t e = mxk::launch_quant_act(x, m, k, static_cast<uint8_t*>(q), static_cast<uint8_t*>(sf), sms,
                                          static_cast<cudaStream_t>(stream), nullptr, true);
    return e == cudaSuccess ? MXFP8_OK : cuda_fail(e);
}

mxfp8_status mxfp8_gemm_128x4(const void* qa, const void* sfa, int64_t m, const mxfp8_weight* w, const void* bias,
                              void* y, void* stream) {
    mxfp8_status st = check_weight(w);
    if (st != MXFP8_OK) return st;
    if (w->num_experts != 1 || m < 0 || m > kMaxRows) return MXFP8_ERR_INVALID_ARG;
    if (m == 0) return MXFP8_OK;
    if (!qa || !sfa || !y) return MXFP8_ERR_INVALID_ARG;
    if (!aligned16(qa) || !aligned16(sfa)) return MXFP8_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(y) & 1u) || (reinterpret_cast<uintptr_t>(bias) & 1u))
        return MXFP8_ERR_MISALIGNED;
    int sms = 0;
    if ((st = device_sms(&sms)) != MXFP8_OK) return st;
    mxk::GemmProblem p = make_problem(qa, sfa, m, w, bias, y, nullptr, nullptr);
    p.sf128 = true;
    // Two weight tiles x 176 tokens per CTA tile (the dual kernel, reading
    // the 128x4 scale tiles each token tile touches; three pipeline stages
    // fit, and measured faster than 160-token tiles with four: 449.7 against
    // 466.5 us at 8192^3) whenever that gives every SM a tile, as the 8x4
    // layer does; else persistent tiles on 128-token boundaries: 256 tokens,
    // or 128 for small M.
    mxk::GemmSchedule sch;
    const int64_t pairs = (w->n_pad / 128 + 1) / 2;
    const bool dual = m > 128 && pairs * ((m + 175) / 176) >= sms;
    sch.tokens_per_tile = dual ? 176 : m > 128 ? 256 : 128;
    sch.split_k = 1;
    sch.persistent = true;
    sch.fuse_quant = false;
    sch.pipes = dual ? 2 : 1;
    sch.dual = dual;
    bool enc_fail = false;
    cudaError_t e = mxk::launch_gemm(p, sch, sms, static_cast<cudaStream_t>(stream), &enc_fail);
    return launch_status(e, enc_fail);
}

mxfp8_status mxfp8_linear_128x4(const void* x, int64_t m, const mxfp8_weight* w, const void* bias, void* y,
                                void* workspace, size_t workspace_bytes, void* stream) {
    mxfp8_status st = check_weight(w);
    if (st != MXFP8_OK) return st;
    if (w->num_experts != 1 || m < 0 || m > kMaxRows) return MXFP8_ERR_INVALID_ARG;
    if (m == 0) return MXFP8_OK;
    if (!x || !workspace) return MXFP8_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return MXFP8_ERR_MISALIGNED;
    if (workspace_bytes < mxfp8_linear_128x4_workspace_bytes(m, w->k)) return MXFP8_ERR_WORKSPACE_TOO_SMALL;
    uint8_t* qa = static_cast<uint8_t*>(workspace);
    uint8_t* sfa = qa + ceil_to(m * w->k, 256);
    if ((st = mxfp8_quantize_act_128x4(x, m, w->k, qa, sfa, stream)) != MXFP8_OK) return st;
    return mxfp8_gemm_128x4(qa, sfa, m, w, bias, y, stream);
}

// --------------------------------------------------------------- tactics
namespace {
// {tokens_per_tile (144/160/176/192 = two weight tiles), split_k (-1 = persistent),
//  fuse_quant, pipes}
void encode_tactic(const mxk::GemmSchedule& s, int32_t* t4) {
    t4[0] = s.tokens_per_tile;
    t4[1] = s.persistent ? -1 : s.split_k;
    t4[2] = s.fuse_quant ? 1 : 0;
    t4[3] = s.dual ? 2 : s.pipes;  // the dual kernel always runs two MMA issuers
}
bool decode_tactic(const int32_t* t4, int kind, int64_t k, mxk::GemmSchedule* s) {
    s->dual = (t4[0] == 192 || t4[0] == 176 || t4[0] == 160 || t4[0] == 144) && t4[1] == -1;
    s->tokens_per_tile = t4[0];
    s->persistent = t4[1] == -1;
    s->split_k = s->persistent ? 1 : t4[1];
    s->fuse_quant = t4[2] != 0;
    s->pipes = t4[3];
    if (s->dual) return t4[1] == -1 && !s->fuse_quant && mxk::schedule_valid(*s, kind, k);
    return mxk::schedule_valid(*s, kind, k);
}
bool kind_ok(int kind) { return kind >= mxk::kTacticLinear && kind <= mxk::kTacticGated; }
}  // namespace

static mxfp8_status autotune_common(const void* x, int64_t m, const int32_t* offsets, const mxfp8_weight* w,
                                    const void* bias, void* y, void* workspace, size_t workspace_bytes, int iters,
                                    void* stream, int32_t* chosen) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return cuda_fail(e);
    if (cap != cudaStreamCaptureStatusNone) return MXFP8_ERR_INVALID_ARG;  // tuning synchronizes
    // One ordinary call validates every argument (and warms the caches).
    mxfp8_status st = linear_common(x, m, offsets, w, bias, y, workspace, workspace_bytes, stream);
    if (st != MXFP8_OK || m == 0) return st;
    if (iters <= 0) iters = 20;
    const int kind = offsets ? mxk::kTacticGrouped : mxk::kTacticLinear;
    const std::vector<mxk::GemmSchedule> cands = mxk::candidate_schedules(kind, m, w->k);
    // Each candidate is timed as one CUDA graph of `iters` back-to-back calls
    // (the way a serving loop replays them): no host launch latency inside
    // the timed region, which would otherwise favour candidates with fewer
    // launches.  The graphs are captured on a private stream that first
    // waits for the caller's.
    cudaStream_t ts = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if ((e = cudaStreamCreateWithFlags(&ts, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaEventCreate(&e0)) != cudaSuccess || (e = cudaEventCreate(&e1)) != cudaSuccess ||
        (e = cudaEventRecord(e0, s)) != cudaSuccess || (e = cudaStreamWaitEvent(ts, e0, 0)) != cudaSuccess) {
        if (e0) cudaEventDestroy(e0);
        if (e1) cudaEventDestroy(e1);
        if (ts) cudaStreamDestroy(ts);
        return cuda_fail(e);
    }
    // A weight smaller than twice the L2 would be served from L2 by calls
    // back to back on one copy; the tuning graphs then rotate over enough
    // temporary copies of it that every call streams its weight from HBM, as
    // the layers of a model do.  Copies that cannot be allocated are left
    // out (the tuning then runs on fewer).
    std::vector<mxfp8_weight> wv(1, *w);
    std::vector<void*> extra;
    {
        int dev = 0, l2 = 0;
        const size_t qb = static_cast<size_t>(w->num_experts * w->n_pad * w->k), sb = qb / 32;
        if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) == cudaSuccess &&
            qb + sb < 2 * static_cast<size_t>(l2)) {
            const int want = std::min<int>(64, static_cast<int>(2 * static_cast<size_t>(l2) / (qb + sb)) + 1);
            for (int c = 1; c < want; ++c) {
                void* q = nullptr;
                void* f = nullptr;
                if (cudaMalloc(&q, qb) != cudaSuccess || cudaMalloc(&f, sb) != cudaSuccess) {
                    if (q) cudaFree(q);
                    (void)cudaGetLastError();
                    break;
                }
                extra.push_back(q);
                extra.push_back(f);
                mxfp8_weight wc = *w;
                wc.q = q;
                wc.sf = f;
                if ((e = cudaMemcpyAsync(q, w->q, qb, cudaMemcpyDeviceToDevice, ts)) != cudaSuccess ||
                    (e = cudaMemcpyAsync(f, w->sf, sb, cudaMemcpyDeviceToDevice, ts)) != cudaSuccess)
                    break;
                wv.push_back(wc);
            }
        }
    }
    int best = -1;
    float best_ms = 0.0f;
    for (size_t i = 0; i < cands.size() && e == cudaSuccess; ++i) {
        t_override = &cands[i];
        bool ok = true;
        for (int r = 0; r < 2 && ok; ++r)
            ok = linear_common(x, m, offsets, w, bias, y, workspace, workspace_bytes, ts) == MXFP8_OK;
        if (!ok) {  // this shape rejects the candidate at launch (resources): skip it
            (void)cudaGetLastError();
            continue;
        }
        cudaGraph_t graph = nullptr;
        cudaGraphExec_t exec = nullptr;
        if ((e = cudaStreamBeginCapture(ts, cudaStreamCaptureModeThreadLocal)) != cudaSuccess) break;
        for (int r = 0; r < iters && ok; ++r)
            ok = linear_common(x, m, offsets, &wv[r % wv.size()], bias, y, workspace, workspace_bytes, ts) == MXFP8_OK;
        const cudaError_t ec = cudaStreamEndCapture(ts, &graph);
        if (!ok || ec != cudaSuccess || cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) {
            (void)cudaGetLastError();  // a candidate the capture rejected: skip it
            if (graph) cudaGraphDestroy(graph);
            continue;
        }
        // One warm launch, then the best of three timed ones.
        float ms = -1.0f;
        e = cudaGraphLaunch(exec, ts);
        for (int rep = 0; rep < 3 && e == cudaSuccess; ++rep) {
            float t = 0.0f;
            if ((e = cudaEventRecord(e0, ts)) == cudaSuccess && (e = cudaGraphLaunch(exec, ts)) == cudaSuccess &&
                (e = cudaEventRecord(e1, ts)) == cudaSuccess && (e = cudaEventSynchronize(e1)) == cudaSuccess &&
                cudaEventElapsedTime(&t, e0, e1) == cudaSuccess && (ms < 0.0f || t < ms))
                ms = t;
        }
        if (e == cudaSuccess && ms >= 0.0f && (best < 0 || ms < best_ms)) {
            best = static_cast<int>(i);
            best_ms = ms;
        }
        cudaGraphExecDestroy(exec);
        cudaGraphDestroy(graph);
    }
    t_override = nullptr;
    const cudaError_t es = cudaStreamSynchronize(ts);
    if (e == cudaSuccess) e = es;
    cudaStreamDestroy(ts);
    for (void* b : extra) cudaFree(b);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (e != cudaSuccess) return cuda_fail(e);
    if (best < 0) return MXFP8_ERR_INVALID_ARG;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e);
    mxk::tactic_store(dev, kind, m, w->n, w->k, w->num_experts, cands[best]);
    if (chosen) encode_tactic(cands[best], chosen);
    return MXFP8_OK;
}

mxfp8_status mxfp8_autotune_linear(const void* x, int64_t m, const mxfp8_weight* w, const void* bias, void* y,
                                   void* workspace, size_t workspace_bytes, int iters, void* stream,
                                   int32_t* chosen) {
    if (w && w->num_experts != 1) return MXFP8_ERR_INVALID_ARG;
    return autotune_common(x, m, nullptr, w, bias, y, workspace, workspace_bytes, iters, stream, chosen);
}

mxfp8_status mxfp8_autotune_grouped_linear(const void* x_sorted, int64_t rows, const int32_t* expert_offsets,
                                           const mxfp8_weight* w, const void* bias, void* y, void* workspace,
                                           size_t workspace_bytes, int iters, void* stream, int32_t* chosen) {
    if (!expert_offsets) return MXFP8_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(expert_offsets) & 3u)) return MXFP8_ERR_MISALIGNED;
    return autotune_common(x_sorted, rows, expert_offsets, w, bias, y, workspace, workspace_bytes, iters, stream,
                           chosen);
}

mxfp8_status mxfp8_tactic_get(int kind, int64_t m, int64_t n, int64_t k, int64_t experts, int32_t* tactic) {
    if (!kind_ok(kind) || m < 1 || n < 1 || k < 1 || experts < 1 || !tactic) return MXFP8_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;  // table operations need no device
    mxk::GemmSchedule s;
    if (!mxk::tactic_lookup(dev, kind, m, n, k, experts, &s)) return MXFP8_ERR_INVALID_ARG;
    encode_tactic(s, tactic);
    return MXFP8_OK;
}

mxfp8_status mxfp8_tactic_set(int kind, int64_t m, int64_t n, int64_t k, int64_t experts, const int32_t* tactic) {
    if (!kind_ok(kind) || m < 1 || n < 1 || k < 1 || k % 256 != 0 || experts < 1 || !tactic)
        return MXFP8_ERR_INVALID_ARG;
    mxk::GemmSchedule s;
    if (!decode_tactic(tactic, kind, k, &s)) return MXFP8_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;  // table operations need no device
    mxk::tactic_store(dev, kind, m, n, k, experts, s);
    return MXFP8_OK;
}

mxfp8_status mxfp8_plan_tactic(int kind, int64_t m, int64_t n, int64_t k, int64_t experts, int sms,
                               int32_t* tactic) {
    const bool grouped = kind == mxk::kTacticGrouped || kind == mxk::kTacticGated;
    if (!kind_ok(kind) || m < 1 || m > kMaxRows || n < 1 || k < 1 || k > kMaxK || experts < 1 ||
        experts > 1024 || !tactic)
        return MXFP8_ERR_INVALID_ARG;
    if (k % 256 != 0) return MXFP8_ERR_K_NOT_MULTIPLE_OF_256;
    if ((!grouped && experts != 1) || (kind == mxk::kTacticGated && n % 128 != 0))
        return MXFP8_ERR_INVALID_ARG;
    if (sms <= 0) {
        mxfp8_status st = device_sms(&sms);
        if (st != MXFP8_OK) return st;
    }
    // Only the presence of x (fusable quantization) and of offsets (grouped)
    // matters to the choice; this marker is never dereferenced.
    alignas(16) static const int32_t kPresent[4] = {0, 0, 0, 0};
    mxk::GemmProblem p{};
    p.m = m;
    p.experts = experts;
    p.n = n;
    p.n_pad = ceil_to(n, 128);
    p.k = k;
    p.offsets = grouped ? kPresent : nullptr;
    p.x = kind == mxk::kTacticLinear ? kPresent : nullptr;
    p.gated = kind == mxk::kTacticGated;
    p.sf128 = false;
    p.hq = nullptr;
    p.hsf = nullptr;
    encode_tactic(select_schedule(p, sms, kind), tactic);
    return MXFP8_OK;
}

void mxfp8_tactic_clear(void) { mxk::tactic_clear(); }

int64_t mxfp8_tactic_count(void) { return mxk::tactic_count(); }

// ------------------------------------------------------------------- MoE
size_t mxfp8_moe_route_workspace_bytes(int64_t tokens, int64_t experts, int64_t topk) {
    if (tokens < 0 || tokens > kMaxRows || experts < 1 || experts > 1024 || topk < 1 || topk > 16) return 0;
    return static_cast<size_t>(((tokens + 7) / 8 * experts + tokens * topk) * 4);  // 8-token routing groups
}

static mxfp8_status check_route_shape(int64_t tokens, int64_t experts, int64_t topk) {
    if (tokens < 0 || topk < 1 || topk > 16 || experts < topk || experts > 1024) return MXFP8_ERR_INVALID_ARG;
    if (tokens * topk >= (int64_t(1) << 31)) return MXFP8_ERR_INVALID_ARG;
    return MXFP8_OK;
}

// release: the routing kernel may release the next kernel once its own
// dependency wait has returned (only the MoE layer, whose next kernel is the
// scattering quantizer).
static mxfp8_status route_checked(const float* logits, int64_t tokens, int64_t experts, int64_t topk,
                                  mxfp8_route_method method, int32_t* topk_ids, float* topk_weights,
                                  int32_t* expert_offsets, int32_t* sorted_token, int32_t* row_of, void* ws,
                                  size_t ws_bytes, void* stream, bool release) {
    mxfp8_status st = check_route_shape(tokens, experts, topk);
    if (st != MXFP8_OK) return st;
    if (method != MXFP8_ROUTE_RENORMALIZE && method != MXFP8_ROUTE_RENORMALIZE_NAIVE) return MXFP8_ERR_INVALID_ARG;
    if (tokens == 0) return MXFP8_OK;
    if (!logits || !topk_ids || !topk_weights || !expert_offsets || !sorted_token || !row_of || !ws)
        return MXFP8_ERR_INVALID_ARG;
    const void* ptrs[] = {logits, topk_ids, topk_weights, expert_offsets, sorted_token, row_of, ws};
    for (const void* q : ptrs)
        if (reinterpret_cast<uintptr_t>(q) & 3u) return MXFP8_ERR_MISALIGNED;
    if (ws_bytes < mxfp8_moe_route_workspace_bytes(tokens, experts, topk)) return MXFP8_ERR_WORKSPACE_TOO_SMALL;
    int sms = 0;
    if ((st = device_sms(&sms)) != MXFP8_OK) return st;
    cudaError_t e = mxk::launch_moe_route(logits, tokens, experts, topk, static_cast<int>(method), topk_ids,
                                          topk_weights, expert_offsets, sorted_token, row_of,
                                          static_cast<int32_t*>(ws), static_cast<cudaStream_t>(stream), release);
    return e == cudaSuccess ? MXFP8_OK : cuda_fail(e);
}

mxfp8_status mxfp8_moe_route(const float* logits, int64_t tokens, int64_t experts, int64_t topk,
                             mxfp8_route_method method, int32_t* topk_ids, float* topk_weights,
                             int32_t* expert_offsets, int32_t* sorted_token, int32_t* row_of, void* ws,
                             size_t ws_bytes, void* stream) {
    return route_checked(logits, tokens, experts, topk, method, topk_ids, topk_weights, expert_offsets,
                         sorted_token, row_of, ws, ws_bytes, stream, false);
}

static mxfp8_status check_gated(const mxfp8_weight* w) {
    mxfp8_status st = check_weight(w);
    if (st != MXFP8_OK) return st;
    if (w->n % 128 != 0) return MXFP8_ERR_INVALID_ARG;  // n = 2 I with I % 64 == 0
    return MXFP8_OK;
}

mxfp8_status mxfp8_prepare_gate_up_weight(const void* src, mxfp8_in_dtype dtype, const mxfp8_weight* w,
                                          void* stream) {
    mxfp8_status st = check_gated(w);
    if (st != MXFP8_OK) return st;
    if (!src || (dtype != MXFP8_IN_F32 && dtype != MXFP8_IN_BF16)) return MXFP8_ERR_INVALID_ARG;
    if (!aligned16(src)) return MXFP8_ERR_MISALIGNED;
    int sms = 0;
    if ((st = device_sms(&sms)) != MXFP8_OK) return st;
    cudaError_t e = mxk::launch_prepare_weight(src, dtype == MXFP8_IN_BF16, w->num_experts, w->n, w->n_pad, w->k,
                                               static_cast<uint8_t*>(w->q), static_cast<uint8_t*>(w->sf), sms,
                                               static_cast<cudaStream_t>(stream), w->n / 2);
    return e == cudaSuccess ? MXFP8_OK : cuda_fail(e);
}

size_t mxfp8_moe_gate_up_workspace_bytes(int64_t rows, int64_t k) { return mxfp8_linear_workspace_bytes(rows, k); }

// The expert-sorted rows of x quantized into ws (the layer's tokens scattered
// through row_of, or the gate_up call's rows gathered through sorted_token),
// then GEMM1 with the SwiGLU epilogue: h as BF16 into h, or (hq != null)
// quantized to MXFP8 into hq and its 8x4 scales into hsf.  Arguments checked
// by the callers.
static mxfp8_status gate_up_launch(const void* x, const int32_t* sorted_token, const int32_t* row_of, int64_t tokens,
                                   int64_t topk, int64_t rows, const int32_t* expert_offsets, const mxfp8_weight* w13,
                                   void* h, uint8_t* hq, uint8_t* hsf, void* ws, int sms, cudaStream_t s) {
    uint8_t* qa = static_cast<uint8_t*>(ws);
    uint8_t* sfa = qa + ceil_to(rows * w13->k, 256);
    cudaError_t e = row_of ? mxk::launch_moe_scatter_quant(x, tokens, topk, w13->k, row_of, qa, sfa, sms, s)
                           : mxk::launch_quant_act(x, rows, w13->k, qa, sfa, sms, s, sorted_token);
    if (e != cudaSuccess) return cuda_fail(e);
    mxk::GemmProblem p = make_problem(qa, sfa, rows, w13, nullptr, h, expert_offsets, nullptr);
    p.gated = true;
    p.hq = hq;
    p.hsf = hsf;
    const mxk::GemmSchedule sch = select_schedule(p, sms, mxk::kTacticGated);
    bool enc_fail = false;
    e = mxk::launch_gemm(p, sch, sms, s, &enc_fail);
    return launch_status(e, enc_fail);
}

mxfp8_status mxfp8_moe_gate_up_swiglu(const void* x, const int32_t* sorted_token, int64_t rows,
                                      const int32_t* expert_offsets, const mxfp8_weight* w13, void* h, void* ws,
                                      size_t ws_bytes, void* stream) {
    mxfp8_status st = check_gated(w13);
    if (st != MXFP8_OK) return st;
    if (rows < 0 || rows > kMaxRows) return MXFP8_ERR_INVALID_ARG;
    if (rows == 0) return MXFP8_OK;
    if (!x || !sorted_token || !expert_offsets || !h || !ws) return MXFP8_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(ws) || (reinterpret_cast<uintptr_t>(h) & 1u) ||
        (reinterpret_cast<uintptr_t>(sorted_token) & 3u) || (reinterpret_cast<uintptr_t>(expert_offsets) & 3u))
        return MXFP8_ERR_MISALIGNED;
    if (ws_bytes < mxfp8_moe_gate_up_workspace_bytes(rows, w13->k)) return MXFP8_ERR_WORKSPACE_TOO_SMALL;
    int sms = 0;
    if ((st = device_sms(&sms)) != MXFP8_OK) return st;
    return gate_up_launch(x, sorted_token, nullptr, 0, 0, rows, expert_offsets, w13, h, nullptr, nullptr, ws, sms,
                          static_cast<cudaStream_t>(stream));
}

// slots_ready: row_of and the weights were complete before the kernel ahead
// of the finalize kernel began (the MoE layer: they come from its routing).
static mxfp8_status finalize_checked(const void* y2, const int32_t* row_of, const float* topk_weights,
                                     int64_t tokens, int64_t topk, int64_t hidden, void* out, void* stream,
                                     bool slots_ready) {
    if (tokens < 0 || topk < 1 || topk > 16 || hidden < 8 || hidden % 8 != 0 || hidden > kMaxK)
        return MXFP8_ERR_INVALID_ARG;
    if (tokens * topk >= (int64_t(1) << 31)) return MXFP8_ERR_INVALID_ARG;
    if (tokens == 0) return MXFP8_OK;
    if (!y2 || !row_of || !topk_weights || !out) return MXFP8_ERR_INVALID_ARG;
    if (!aligned16(y2) || !aligned16(out) || (reinterpret_cast<uintptr_t>(row_of) & 3u) ||
        (reinterpret_cast<uintptr_t>(topk_weights) & 3u))
        return MXFP8_ERR_MISALIGNED;
    int sms = 0;
    mxfp8_status st = device_sms(&sms);
    if (st != MXFP8_OK) return st;
    cudaError_t e = mxk::launch_moe_finalize(y2, row_of, topk_weights, tokens, topk, hidden, out, sms,
                                             static_cast<cudaStream_t>(stream), slots_ready);
    return e == cudaSuccess ? MXFP8_OK : cuda_fail(e);
}

mxfp8_status mxfp8_moe_finalize(const void* y2, const int32_t* row_of, const float* topk_weights,
                                int64_t tokens, int64_t topk, int64_t hidden, void* out, void* stream) {
    return finalize_checked(y2, row_of, topk_weights, tokens, topk, hidden, out, stream, false);
}

namespace {
// Sub-buffers of the expert-MLP workspace, each 256-byte aligned.
struct MoeWs {
    size_t ids, weights, offsets, sorted_token, row_of, route, g1, h, g2, y2, total;
};
MoeWs moe_layout(int64_t tokens, int64_t experts, int64_t topk, int64_t hidden, int64_t inter) {
    const int64_t r = tokens * topk;
    MoeWs l;
    size_t at = 0;
    auto take = [&](size_t bytes) { const size_t p = at; at += static_cast<size_t>(ceil_to(bytes, 256)); return p; };
    l.ids = take(r * 4);
    l.weights = take(r * 4);
    l.offsets = take((experts + 1) * 4);
    l.sorted_token = take(r * 4);
    l.row_of = take(r * 4);
    l.route = take(mxfp8_moe_route_workspace_bytes(tokens, experts, topk));
    l.g1 = take(mxfp8_linear_workspace_bytes(r, hidden));
    l.h = take(r * inter * 2);
    l.g2 = take(mxfp8_linear_workspace_bytes(r, inter));
    l.y2 = take(r * hidden * 2);
    l.total = at;
    return l;
}
}  // namespace

size_t mxfp8_moe_workspace_bytes(int64_t tokens, int64_t experts, int64_t topk, int64_t hidden, int64_t inter) {
    if (check_route_shape(tokens, experts, topk) != MXFP8_OK || hidden <= 0 || inter <= 0 || hidden % 32 ||
        inter % 32 || hidden > kMaxK || inter > kMaxK)
        return 0;
    return moe_layout(tokens, experts, topk, hidden, inter).total;
}

mxfp8_status mxfp8_moe_expert_mlp(const void* x, const float* logits, int64_t tokens, int64_t topk,
                                  mxfp8_route_method method, const mxfp8_weight* w13, const mxfp8_weight* w2,
                                  void* out, void* ws, size_t ws_bytes, void* stream) {
    mxfp8_status st = check_gated(w13);
    if (st != MXFP8_OK) return st;
    if ((st = check_weight(w2)) != MXFP8_OK) return st;
    const int64_t experts = w13->num_experts, hidden = w13->k, inter = w13->n / 2;
    if (w2->num_experts != experts || w2->n != hidden || w2->k != inter) return MXFP8_ERR_INVALID_ARG;
    if ((st = check_route_shape(tokens, experts, topk)) != MXFP8_OK) return st;
    if (tokens == 0) return MXFP8_OK;
    if (!x || !logits || !out || !ws) return MXFP8_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out) || !aligned16(ws) || (reinterpret_cast<uintptr_t>(logits) & 3u))
        return MXFP8_ERR_MISALIGNED;
    const MoeWs l = moe_layout(tokens, experts, topk, hidden, inter);
    if (ws_bytes < l.total) return MXFP8_ERR_WORKSPACE_TOO_SMALL;
    uint8_t* b = static_cast<uint8_t*>(ws);
    int32_t* ids = reinterpret_cast<int32_t*>(b + l.ids);
    float* wts = reinterpret_cast<float*>(b + l.weights);
    int32_t* off = reinterpret_cast<int32_t*>(b + l.offsets);
    int32_t* stok = reinterpret_cast<int32_t*>(b + l.sorted_token);
    int32_t* row_of = reinterpret_cast<int32_t*>(b + l.row_of);
    const int64_t r = tokens * topk;
    int sms = 0;
    if ((st = device_sms(&sms)) != MXFP8_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // GEMM1's SwiGLU epilogue writes h already quantized (E4M3 + 8x4 scales,
    // the bytes the activation quantizer would make of the BF16 h) into the
    // GEMM2 activation buffers, so GEMM2 runs on them directly.
    uint8_t* hq = b + l.g2;
    uint8_t* hsf = hq + ceil_to(r * inter, 256);
    if (r % 8 != 0) {
        // Rows r..ceil8(r)-1 of h's last 8-row scale group hold 0x00, as the
        // quantizer writes them: clear that group (before routing, so that the
        // router's next kernel is the gathering quantizer); GEMM1 then fills
        // rows < r.
        const int64_t grp = ceil_to(inter / 32, 4) * 8;
        cudaError_t e = cudaMemsetAsync(hsf + (r / 8) * grp, 0, static_cast<size_t>(grp), s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    // The router releases the scattering quantizer once its own dependency
    // wait has returned (x is then complete): the quantizer loads and
    // quantizes x while the router runs, waits for it, scatters the rows
    // through row_of and releases GEMM1, which reads the offsets in its
    // prologue.
    st = route_checked(logits, tokens, experts, topk, method, ids, wts, off, stok, row_of, b + l.route,
                       mxfp8_moe_route_workspace_bytes(tokens, experts, topk), stream, true);
    if (st != MXFP8_OK) return st;
    st = gate_up_launch(x, nullptr, row_of, tokens, topk, r, off, w13, nullptr, hq, hsf, b + l.g1, sms, s);
    if (st != MXFP8_OK) return st;
    mxk::GemmProblem p2 = make_problem(hq, hsf, r, w2, nullptr, b + l.y2, off, nullptr);
    const mxk::GemmSchedule sch2 = select_schedule(p2, sms, mxk::kTacticGrouped);
    bool enc_fail = false;
    cudaError_t e = mxk::launch_gemm(p2, sch2, sms, s, &enc_fail);
    if ((st = launch_status(e, enc_fail)) != MXFP8_OK) return st;
    return finalize_checked(b + l.y2, row_of, wts, tokens, topk, hidden, out, stream, true);
}

const char* mxfp8_status_string(mxfp8_status s) {
    switch (s) {
        case MXFP8_OK: return "ok";
        case MXFP8_ERR_INVALID_ARG: return "invalid argument";
        case MXFP8_ERR_K_NOT_MULTIPLE_OF_256: return "K must be a multiple of 256";
        case MXFP8_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
        case MXFP8_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3 (GB300)";
        case MXFP8_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case MXFP8_ERR_DEVICE_TIMEOUT: return "a kernel gave up waiting (device timeout)";
        case MXFP8_ERR_CUDA: return "CUDA error (see mxfp8_last_cuda_error)";
        case MXFP8_ERR_OUT_OF_BOUNDS: return "a kernel computed a store index outside its buffer (debug build)";
    }
    return "unknown status";
}

int mxfp8_last_cuda_error(void) { return t_last_cuda_error; }

mxfp8_status mxfp8_device_error(void) {
    unsigned int v = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    e = mxk::read_and_clear_gemm_error(&v);
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned int oob = 0, w = 0;
    if ((e = mxk::read_and_clear_oob_gemm(&w)) != cudaSuccess) return cuda_fail(e);
    oob |= w;
    if ((e = mxk::read_and_clear_oob_quant(&w)) != cudaSuccess) return cuda_fail(e);
    oob |= w;
    if ((e = mxk::read_and_clear_oob_moe(&w)) != cudaSuccess) return cuda_fail(e);
    oob |= w;
    if (v) return MXFP8_ERR_DEVICE_TIMEOUT;
    return oob ? MXFP8_ERR_OUT_OF_BOUNDS : MXFP8_OK;
}

int mxfp8_debug_build(void) {
#ifdef MXFP8_DEBUG
    return 1;
#else
    return 0;
#endif
}

void mxfp8_set_wait_limit_ns(uint64_t ns) { mxk::set_wait_limit_ns(ns); }

void mxfp8_set_pipes(int pipes) { mxk::set_pipes(pipes); }

void mxfp8_last_schedule(int* out5) {
    if (out5) mxk::last_schedule(out5);
}

void mxfp8_set_schedule(int tokens_per_tile, int split_k, int fuse_quant) {
    // 144 / 160 / 176 / 192: the dual weight-tile schedule (dense, persistent).
    const bool tt_ok = tokens_per_tile == 0 || tokens_per_tile == 16 || tokens_per_tile == 32 ||
                       tokens_per_tile == 64 || tokens_per_tile == 128 || tokens_per_tile == 256 ||
                       tokens_per_tile == 144 || tokens_per_tile == 160 || tokens_per_tile == 176 ||
                       tokens_per_tile == 192;
    g_force_tt.store(tt_ok ? tokens_per_tile : 0, std::memory_order_relaxed);
    g_force_split.store((split_k >= -1 && split_k <= 8) ? split_k : 0, std::memory_order_relaxed);
    g_force_fuse.store((fuse_quant >= -1 && fuse_quant <= 1) ? fuse_quant : -1, std::memory_order_relaxed);
}

}  // extern "C"
