// internal.h -- host-side interfaces between the C ABI (api.cu) and the
// kernel translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

namespace mxk {

// Activation quantizer, 8x4 scale layout.  It lets a dependent grid launched
// with programmatic stream serialization start its prologue early.  With
// src_rows, output row r quantizes input row src_rows[r].
cudaError_t launch_quant_act(const void* x, int64_t m, int64_t k, uint8_t* q, uint8_t* sf,
                             int num_sms, cudaStream_t s, const int32_t* src_rows = nullptr,
                             bool layout_128x4 = false);

// Weight preparation: quantize + pad N + prepared layout.  src_is_bf16
// selects the element type of src ([experts][n][k]); inter > 0 applies the
// gated-row reorder of GEMM1 weights [gate; up] with n = 2 * inter.
cudaError_t launch_prepare_weight(const void* src, bool src_is_bf16, int64_t experts, int64_t n,
                                  int64_t n_pad, int64_t k, uint8_t* q, uint8_t* sf, int num_sms,
                                  cudaStream_t s, int64_t inter = 0);

// Mixture-of-experts helpers (moe.cu).  Routing: top-k per token, weights,
// and the stable expert-sorted order; ws holds ceil(tokens/8) * experts
// group counts plus tokens * topk ranks (int32).
cudaError_t launch_moe_route(const float* logits, int64_t tokens, int64_t experts, int64_t topk, int method,
                             int32_t* ids, float* weights, int32_t* offsets, int32_t* sorted_token,
                             int32_t* row_of, int32_t* ws, cudaStream_t s, bool release = false);
// MoE GEMM1's activations by token: x (BF16 [tokens][k], k a multiple of 128)
// quantized once per token and written to rows row_of[t * topk + s] of qa
// (E4M3 [tokens*topk][k]) with 8x4 scales in sfa (pad rows' scales zero).
// Reads x before its dependency wait: the kernel ahead must release it only
// once x is complete.
cudaError_t launch_moe_scatter_quant(const void* x, int64_t tokens, int64_t topk, int64_t k, const int32_t* row_of,
                                     uint8_t* qa, uint8_t* sfa, int num_sms, cudaStream_t s);
// out[t] = bf16(sum_s weights[t, s] * y2[row_of[t * topk + s]]), FP32 sum in slot order.
// slots_ready: row_of and weights were complete before the kernel this one
// depends on began (they may then be read before the dependency wait).
cudaError_t launch_moe_finalize(const void* y2, const int32_t* row_of, const float* weights, int64_t tokens,
                                int64_t topk, int64_t hidden, void* out, int num_sms, cudaStream_t s,
                                bool slots_ready = false);

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
    const void* x;             // bf16 [m][k] activations when the GEMM may quantize them itself
    bool gated;                // grouped only: SwiGLU epilogue, y = silu(gate) * up, bf16 [m][n/2]
    uint8_t* hq;               // gated only, or null: write h quantized to MXFP8 instead of BF16 y:
    uint8_t* hsf;              //   E4M3 [m][n/2] and its 8x4 scales (rows past m untouched)
    bool sf128;                // sfa uses the 128x4 layout (dense, persistent tiles of 128/256 tokens)
};

struct GemmSchedule {
    int tokens_per_tile;       // 16, 32, 64, 128, 256
    int split_k;               // CTAs (a cluster) per output tile, K split among them
    bool persistent;           // tiles strided over a persistent grid (split_k == 1)
    bool fuse_quant;           // the GEMM quantizes x itself (one-tile schedules)
    int pipes;                 // MMA pipelines per CTA (1, 2 or 4; >1 only for <= 64 tokens)
    bool dual;                 // dense, persistent, two weight tiles x 192 tokens per CTA tile
};

// Tactic table (tactics.cu).  Kinds of calls with separate entries.
constexpr int kTacticLinear = 0;   // mxfp8_linear: x available, quantization may be fused
constexpr int kTacticGemm = 1;     // mxfp8_gemm: pre-quantized activations
constexpr int kTacticGrouped = 2;  // mxfp8_grouped_linear
constexpr int kTacticGated = 3;    // MoE GEMM1 with the SwiGLU epilogue
int64_t m_bucket(int64_t m);       // smallest power of two >= m
bool schedule_valid(const GemmSchedule& s, int kind, int64_t k);
bool tactic_lookup(int dev, int kind, int64_t m, int64_t n, int64_t k, int64_t experts, GemmSchedule* out);
void tactic_store(int dev, int kind, int64_t m, int64_t n, int64_t k, int64_t experts, const GemmSchedule& s);
void tactic_clear();
int64_t tactic_count();
std::vector<GemmSchedule> candidate_schedules(int kind, int64_t m, int64_t k);

// Testing hook: pipelines per CTA for later launches (0 = automatic).
void set_pipes(int pipes);

// force_tt: 0 or a token tile; force_split: 0 auto, -1 persistent, >0 split;
// force_fuse: -1 auto, 0 off, 1 on where possible.
GemmSchedule choose_schedule(const GemmProblem& p, int num_sms, int force_tt, int force_split,
                             int force_fuse);

// Returns cudaSuccess or the launch/encode error; sets *encode_failed when a
// tensor map could not be encoded (reported as an invalid argument).
cudaError_t launch_gemm(const GemmProblem& p, const GemmSchedule& sch, int num_sms,
                        cudaStream_t s, bool* encode_failed);

// Schedule of this thread's last GEMM launch: {tokens per tile, split (-1 =
// persistent), fused quantization, grid, stages}.
void last_schedule(int* out5);

// Limit of every pipeline wait of later GEMM launches (0 = the default).
void set_wait_limit_ns(uint64_t ns);

// Records a failed CUDA call's code for mxfp8_last_cuda_error() (this thread).
void record_cuda_error(int e);

// Reads and clears the device error word of the GEMM kernels.
cudaError_t read_and_clear_gemm_error(unsigned int* out);

// Read and clear the out-of-bounds-store words of the debug build (one per
// kernel translation unit; always 0 in the normal build).
cudaError_t read_and_clear_oob_gemm(unsigned int* out);
cudaError_t read_and_clear_oob_quant(unsigned int* out);
cudaError_t read_and_clear_oob_moe(unsigned int* out);

}  // namespace mxk
