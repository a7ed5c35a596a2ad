// noalloc.cu -- mxfp8_linear for callers that cannot allocate device memory.
//
// Some callers have no way to provide the workspace that mxfp8_linear needs:
// code embedded in a host framework that owns every device allocation (a
// cudaMalloc behind its back would break its memory accounting), or serving
// paths that must never allocate once they are running.  For them this file
// keeps the activation scratch in a fixed device array of the library.  The
// array is a file-scope __device__ variable, so every GPU that loads the
// library holds MXFP8_STATIC_SCRATCH_BYTES of it until the process exits.
//
// The path is the unfused one of mxfp8_linear: the activation quantizer writes
// the E4M3 bytes and the 8x4 scales into the array, then the block-scaled GEMM
// reads them.  Every byte the GEMM reads is written by the quantizer of the
// same call, so nothing has to be cleared between calls; the array keeps the
// last call's contents.  All calls share the one array: calls whose kernels
// overlap on the GPU (different streams, different threads) race on it and
// must be serialised by the caller.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/mxfp8.h"
#include "internal.h"

namespace {

__device__ __align__(256) uint8_t g_static_scratch[MXFP8_STATIC_SCRATCH_BYTES];

struct ScratchSlot {
    bool ready;
    uint8_t* ptr;  // device address of g_static_scratch on that device
    int sms;
};
ScratchSlot g_slot[64];
std::mutex g_slot_mu;
thread_local int t_static_cuda_error = 0;

// A failed CUDA call: its code goes to both mxfp8_static_scratch_last_cuda_error()
// and mxfp8_last_cuda_error(), as for every other entry point.
mxfp8_status cuda_error(cudaError_t e) {
    t_static_cuda_error = static_cast<int>(e);
    mxk::record_cuda_error(static_cast<int>(e));
    return MXFP8_ERR_CUDA;
}

int64_t round_up(int64_t v, int64_t q) { return (v + q - 1) / q * q; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Once per device, with that device current: the array's device address.  The
// name g_static_scratch in host code is only a host-side stand-in.
mxfp8_status scratch_for_current_device(uint8_t** ptr, int* sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e);
    if (dev < 0 || dev >= 64) return MXFP8_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_slot_mu);
    ScratchSlot& s = g_slot[dev];
    if (!s.ready) {
        int major = 0, minor = 0, count = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_error(e);
        if (major != 10 || minor != 3) return MXFP8_ERR_UNSUPPORTED_DEVICE;
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || p == nullptr) return cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
        s.ptr = static_cast<uint8_t*>(p);
        s.sms = count;
        s.ready = true;
    }
    *ptr = s.ptr;
    *sms = s.sms;
    return MXFP8_OK;
}

}  // namespace

extern "C" mxfp8_status mxfp8_linear_static_scratch(const void* x, int64_t m, const mxfp8_weight* w,
                                                    const void* bias, void* y, void* stream) {
    if (!w || !w->q || !w->sf || w->num_experts != 1 || w->n < 1) return MXFP8_ERR_INVALID_ARG;
    if (w->k < 1 || w->k % 256 != 0) return w->k < 1 ? MXFP8_ERR_INVALID_ARG : MXFP8_ERR_K_NOT_MULTIPLE_OF_256;
    if (w->n_pad != round_up(w->n, 128) || w->k > (int64_t(1) << 20) || w->n_pad > (int64_t(1) << 30))
        return MXFP8_ERR_INVALID_ARG;
    if (m < 0) return MXFP8_ERR_INVALID_ARG;
    if (m == 0) return MXFP8_OK;
    if (!x || !y) return MXFP8_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w->q, 16) || !aligned(w->sf, 16) || !aligned(y, 2) ||
        (bias && !aligned(bias, 2)))
        return MXFP8_ERR_MISALIGNED;
    // The quantized activations and their 8x4 scales must fit the array.
    if (m > (int64_t(1) << 30) / w->k) return MXFP8_ERR_WORKSPACE_TOO_SMALL;
    const int64_t q_bytes = round_up(m * w->k, 256);
    const int64_t sf_bytes = round_up(m, 8) * (w->k / 32);
    if (q_bytes + sf_bytes > static_cast<int64_t>(MXFP8_STATIC_SCRATCH_BYTES)) return MXFP8_ERR_WORKSPACE_TOO_SMALL;

    uint8_t* scratch = nullptr;
    int sms = 0;
    mxfp8_status st = scratch_for_current_device(&scratch, &sms);
    if (st != MXFP8_OK) return st;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* qa = scratch;
    uint8_t* sfa = scratch + q_bytes;
    cudaError_t e = mxk::launch_quant_act(x, m, w->k, qa, sfa, sms, s);
    if (e != cudaSuccess) return cuda_error(e);

    mxk::GemmProblem p;
    p.qa = qa;
    p.sfa = sfa;
    p.m = m;
    p.wq = static_cast<const uint8_t*>(w->q);
    p.wsf = static_cast<const uint8_t*>(w->sf);
    p.experts = 1;
    p.n = w->n;
    p.n_pad = w->n_pad;
    p.k = w->k;
    p.bias = bias;
    p.y = y;
    p.offsets = nullptr;
    p.x = nullptr;  // the GEMM reads the quantized activations from the array
    p.gated = false;
    p.sf128 = false;
    p.hq = nullptr;
    p.hsf = nullptr;
    // The schedule of an unfused mxfp8_linear call of this class: a stored
    // tactic if the table holds an unfused one for it, else the built-in
    // heuristic with quantization not fused.
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_error(e);
    mxk::GemmSchedule sch;
    if (!mxk::tactic_lookup(dev, mxk::kTacticLinear, m, w->n, w->k, 1, &sch) || sch.fuse_quant)
        sch = mxk::choose_schedule(p, sms, 0, 0, 0);
    bool enc_fail = false;
    e = mxk::launch_gemm(p, sch, sms, s, &enc_fail);
    if (enc_fail) return MXFP8_ERR_INVALID_ARG;
    if (e != cudaSuccess) return cuda_error(e);
    return MXFP8_OK;
}

extern "C" int mxfp8_static_scratch_last_cuda_error(void) { return t_static_cuda_error; }
