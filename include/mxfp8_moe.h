/*
 * mxfp8_moe.h -- C ABI of the MXFP8 mixture-of-experts expert MLP on GB300.
 *
 * One MoE layer, as the FlashInfer pages describe it:
 *   FlashInfer PR #1214 "TRT-LLM Gen MoE" (Highlights): two routing methods,
 *   Renormalize (top-k of the logits, then a softmax over those k) and
 *   RenormalizeNaive (a softmax over all experts, the top-k, then the k picks
 *   rescaled to sum to 1); the GEMM1 weight rows are reordered for the gated
 *   activation during weight preparation.  The unified-MoE per-tensor FP8 PR
 *   (What changed): GEMM1 (gate/linear) then GEMM2, with the gated-row
 *   reorder of GEMM1.
 * The steps of mxfp8_moe_expert_mlp:
 *   1. route: per token the top-k experts and their weights, then the
 *      (token, slot) pairs sorted by expert, then token;
 *   2. gate_up: the token rows in expert-sorted order, quantized (MXFP8,
 *      8x4 scales; inside mxfp8_moe_expert_mlp each token is quantized once
 *      and written to its top-k rows, the gate_up call gathers rows through
 *      sorted_token: the same bytes), grouped GEMM1 against the gated weights
 *      and the SwiGLU epilogue h = silu(gate) * up, rounded to BF16 [rows][I];
 *   3. down: grouped GEMM2 of h into BF16 [rows][H].  Inside
 *      mxfp8_moe_expert_mlp, GEMM1's epilogue quantizes the BF16 h straight
 *      to MXFP8 (8x4 scales) for GEMM2; run as separate calls,
 *      mxfp8_moe_gate_up_swiglu writes the BF16 h and mxfp8_grouped_linear
 *      quantizes it: the same bytes either way;
 *   4. finalize: out[t] = sum over slots s of w[t,s] * down[row(t,s)] (FP32
 *      in slot order, one BF16 rounding).
 * Readings taken where the pages are silent: the gated activation is SwiGLU
 * (silu(g) = g / (1 + exp(-g))) on GEMM1 rows [gate; up]; experts are chosen
 * on the raw logits (equal to choosing on the softmax in exact arithmetic),
 * descending, ties to the lower expert id; the intermediate h is BF16; no
 * bias.
 *
 * Conventions are those of mxfp8.h (device pointers, caller-owned memory,
 * asynchronous on `stream`, host-side checks before any launch, CUDA-graph
 * capturable, deterministic, GB300 only).  Integer buffers are int32.
 * Limits: 1 <= topk <= 16, topk <= experts <= 1024, tokens * topk < 2^31.
 */
#ifndef MXFP8_GB300_MOE_H
#define MXFP8_GB300_MOE_H

#include "mxfp8.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mxfp8_route_method {
    MXFP8_ROUTE_RENORMALIZE = 0,       /* top-k of the logits, softmax over those k */
    MXFP8_ROUTE_RENORMALIZE_NAIVE = 1  /* softmax over all experts, top-k, renormalize to sum 1 */
} mxfp8_route_method;

/* Workspace of mxfp8_moe_route: (ceil(tokens/8) * experts + tokens * topk)
 * int32. */
size_t mxfp8_moe_route_workspace_bytes(int64_t tokens, int64_t experts, int64_t topk);

/* Routing of `tokens` tokens over `experts` experts.
 * logits: float32 [tokens][experts].  Outputs (device, caller-owned):
 *   topk_ids      int32 [tokens][topk]  experts per token, descending logit
 *   topk_weights  float [tokens][topk]  routing weights (sum to 1 per token)
 *   expert_offsets int32 [experts + 1]  exclusive prefix of per-expert counts
 *   sorted_token  int32 [tokens*topk]   token of each expert-sorted row
 *   row_of        int32 [tokens*topk]   expert-sorted row of pair (t, s) at t*topk + s
 * ws: >= mxfp8_moe_route_workspace_bytes.  Up to 512 tokens one launch does
 * everything (one cluster of 16 CTAs where the GPU schedules it and
 * experts <= 512, else of 8 CTAs, that exchange per-group expert counts
 * through distributed shared memory; ws is then not touched); above, two
 * launches (per-group selection, then one scan over the groups).  The
 * kernel that writes the offsets never releases its programmatic
 * dependents early. */
mxfp8_status mxfp8_moe_route(const float* logits, int64_t tokens, int64_t experts, int64_t topk,
                             mxfp8_route_method method, int32_t* topk_ids, float* topk_weights,
                             int32_t* expert_offsets, int32_t* sorted_token, int32_t* row_of,
                             void* ws, size_t ws_bytes, void* stream);

/* Load-time preparation of GEMM1 weights with the gated-row reorder.
 * src: [num_experts][2*I][k] float32 or bfloat16 (rows [gate; up]); w: a
 * view with n = 2*I, I a multiple of 64.  Prepared 128-row tile j holds
 * gate rows [64j, 64j + 64) then up rows [I + 64j, I + 64j + 64); data and
 * scales otherwise as mxfp8_prepare_weight. */
mxfp8_status mxfp8_prepare_gate_up_weight(const void* src, mxfp8_in_dtype dtype,
                                          const mxfp8_weight* w, void* stream);

/* Workspace of mxfp8_moe_gate_up_swiglu for `rows` sorted rows of k = H:
 * mxfp8_linear_workspace_bytes(rows, k). */
size_t mxfp8_moe_gate_up_workspace_bytes(int64_t rows, int64_t k);

/* Step 2: h[r] = bf16(silu(gate_r) * up_r) for every expert-sorted row r,
 * where [gate_r; up_r] = GEMM1 of expert e (off[e] <= r < off[e+1]) applied
 * to the MXFP8-quantized token row x[sorted_token[r]].
 * x: bfloat16 [tokens][k]; w13: prepared by mxfp8_prepare_gate_up_weight;
 * h: bfloat16 [rows][I] (I = w13->n / 2).
 * sorted_token (int32 [rows]) and expert_offsets (int32 [E + 1]) are read
 * on the device and not checked: every sorted_token value must lie in
 * [0, tokens), and the offsets must follow mxfp8_grouped_linear's rules,
 * including its ordering rule (mxfp8_moe_route's outputs satisfy both; the
 * gathering quantizer this call launches first waits for the kernel before
 * it and only then lets GEMM1 start).
 * ws: >= mxfp8_moe_gate_up_workspace_bytes(rows, k), 16-B aligned. */
mxfp8_status mxfp8_moe_gate_up_swiglu(const void* x, const int32_t* sorted_token, int64_t rows,
                                      const int32_t* expert_offsets, const mxfp8_weight* w13, void* h,
                                      void* ws, size_t ws_bytes, void* stream);

/* Step 4: out[t][c] = bf16( sum_{s < topk} topk_weights[t][s] *
 * y2[row_of[t*topk + s]][c] ), summed in FP32 in slot order.
 * y2: bfloat16 [tokens*topk][hidden]; out: bfloat16 [tokens][hidden];
 * hidden % 8 == 0; y2 and out 16-byte aligned.  row_of values are read on
 * the device and not checked: each must lie in [0, tokens*topk). */
mxfp8_status mxfp8_moe_finalize(const void* y2, const int32_t* row_of, const float* topk_weights,
                                int64_t tokens, int64_t topk, int64_t hidden, void* out, void* stream);

/* Workspace of mxfp8_moe_expert_mlp. */
size_t mxfp8_moe_workspace_bytes(int64_t tokens, int64_t experts, int64_t topk, int64_t hidden,
                                 int64_t inter);

/* The whole expert MLP of one layer: steps 1-4.
 * x: bfloat16 [tokens][H]; logits: float32 [tokens][E];
 * w13: GEMM1 weights (E experts, n = 2I, k = H) from
 * mxfp8_prepare_gate_up_weight; w2: GEMM2 weights (E experts, n = H, k = I)
 * from mxfp8_prepare_weight; out: bfloat16 [tokens][H].
 * Requires H % 256 == 0 and I % 256 == 0 (both are GEMM K dimensions).
 * Launches, each with programmatic dependent launch: routing, the
 * scattering quantizer (released by the router once the router's own wait
 * has returned, so x is complete: it quantizes x while the router runs, then
 * waits for it, writes the rows through the router's row indices and lets
 * GEMM1 start), GEMM1 with the SwiGLU epilogue writing h as MXFP8, GEMM2,
 * finalize (which loads the router's row indices and weights before it waits
 * for GEMM2). */
mxfp8_status mxfp8_moe_expert_mlp(const void* x, const float* logits, int64_t tokens, int64_t topk,
                                  mxfp8_route_method method, const mxfp8_weight* w13,
                                  const mxfp8_weight* w2, void* out, void* ws, size_t ws_bytes,
                                  void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MXFP8_GB300_MOE_H */
