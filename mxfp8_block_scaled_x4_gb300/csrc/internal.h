// internal.h -- host-side interfaces between the C ABI (api.cu) and the
// kernel translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mxk {

// Activation quantizer, 8x4 scale layout.  It lets a dependent grid launched
// with programmatic stream serialization start its prologue early.
cudaError_t launch_quant_act(const void* x, int64_t m, int64_t k, uint8_t* q, uint8_t* sf,
                             int num_sms, cudaStream_t s);

// Weight preparation: quantize + pad N + prepared layout.  src_is_bf16
// selects the element type of src ([experts][n][k]).
cudaError_t launch_prepare_weight(const void* src, bool src_is_bf16, int64_t experts, int64_t n,
                                  int64_t n_pad, int64_t k, uint8_t* q, uint8_t* sf, int num_sms,
                                  cudaStream_t s);

struct GemmProblem {
    const uint8_t* qa;         // [m][k] E4M3 activations
    const uint8_t* sfa;        // 8x4 scales of qa
    int64_t m;                 // activation rows
    const uint8_t* wq;         // [experts][n_pad][k]
    const uint8_t* wsf;        // tiled weight scales
    int64_t experts;
    int64_t n, n_pad, k;
    const void* bias;          // bf16 [experts][n] or null
    void* y;                   // bf16 [m][n]
    const int32_t* offsets;    // grouped: device [experts + 1]; dense: null
    bool after_quant;          // launch as a programmatic dependent of the previous kernel
};

struct GemmSchedule {
    int tokens_per_tile;       // 16, 32, 64, 128, 256
    int split_k;               // 1 = persistent tiles, >1 = cluster split-K
};

GemmSchedule choose_schedule(const GemmProblem& p, int num_sms, int force_tt, int force_split);

// Returns cudaSuccess or the launch/encode error; sets *encode_failed when a
// tensor map could not be encoded (reported as an invalid argument).
cudaError_t launch_gemm(const GemmProblem& p, const GemmSchedule& sch, int num_sms,
                        cudaStream_t s, bool* encode_failed);

// Reads and clears the device error word of the GEMM kernels.
cudaError_t read_and_clear_gemm_error(unsigned int* out);

}  // namespace mxk
