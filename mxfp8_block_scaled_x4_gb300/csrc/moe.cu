// moe.cu -- routing and finalize kernels of the MXFP8 mixture-of-experts
// expert MLP.
//
// Routing follows FlashInfer PR #1214 "TRT-LLM Gen MoE" (Highlights):
// "Renormalize (TopK -> Softmax)" and "RenormalizeNaive (Softmax -> TopK ->
// Renormalize)".  The experts of a token are chosen on the raw logits (the
// softmax is strictly monotone, so this is the top-k of the probabilities in
// exact arithmetic), in descending order, ties to the lower expert id.  The
// (token, slot) pairs are then sorted by expert, then token -- stable and
// deterministic, no atomics:
//   route_topk_kernel   one lane per token: top-k by insertion over the
//                       logits, the weights, and per 32-token group a ballot
//                       per expert -> group counts and each pair's rank
//                       inside its group;
//   route_scan_kernel   one CTA: per-expert totals -> offsets, and per
//                       (group, expert) the first sorted row of that group;
//   route_assign_kernel row_of[t*k + s] and sorted_token[row].
// Finalize sums each token's k expert outputs with its routing weights in
// slot order (FP32) and rounds once to BF16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace mxk {

namespace {

constexpr int kMaxTopK = 16;
constexpr int kRouteThreads = 128;

__global__ void __launch_bounds__(kRouteThreads)
    route_topk_kernel(const float* __restrict__ logits, int tokens, int experts, int topk, int method,
                      int32_t* __restrict__ ids, float* __restrict__ weights,
                      int32_t* __restrict__ grp_count, int32_t* __restrict__ rank) {
    const int lane = threadIdx.x & 31;
    const int group = (blockIdx.x * kRouteThreads + threadIdx.x) >> 5;
    const int t = group * 32 + lane;
    const bool live = t < tokens;
    if (group * 32 >= tokens) return;  // warp-uniform
    float v[kMaxTopK];
    int id[kMaxTopK];
#pragma unroll
    for (int i = 0; i < kMaxTopK; ++i) { v[i] = -INFINITY; id[i] = 0x7FFFFFFF; }
    const float* lg = logits + static_cast<size_t>(live ? t : 0) * experts;
    if (live) {
        // Insertion over ascending expert ids: a new logit goes after every
        // kept entry >= it, so equal logits keep the lower id first.
        for (int e = 0; e < experts; ++e) {
            const float x = lg[e];
            if (!(x > v[topk - 1]) && id[topk - 1] != 0x7FFFFFFF) continue;
#pragma unroll
            for (int i = kMaxTopK - 1; i >= 0; --i) {
                if (i >= topk) continue;
                // Slots x beats move down by one; x lands below the last
                // entry it does not beat.
                const bool beats_here = x > v[i] || id[i] == 0x7FFFFFFF;
                if (!beats_here) continue;
                const bool goes_higher = i > 0 && (x > v[i > 0 ? i - 1 : 0] || id[i > 0 ? i - 1 : 0] == 0x7FFFFFFF);
                if (goes_higher) { v[i] = v[i - 1]; id[i] = id[i - 1]; }
                else { v[i] = x; id[i] = e; }
            }
        }
        // Weights.  m = v[0] is the largest logit of the token.
        float z[kMaxTopK];
        float zs = 0.0f;
#pragma unroll
        for (int i = 0; i < kMaxTopK; ++i) {
            z[i] = i < topk ? expf(v[i] - v[0]) : 0.0f;
            zs += z[i];
        }
        if (method == 1) {
            // Softmax over all logits, then renormalize the selected ones.
            float all = 0.0f;
            for (int e = 0; e < experts; ++e) all += expf(lg[e] - v[0]);
            float ps = 0.0f;
#pragma unroll
            for (int i = 0; i < kMaxTopK; ++i) {
                z[i] = z[i] / all;
                ps += i < topk ? z[i] : 0.0f;
            }
            zs = ps;
        }
#pragma unroll
        for (int i = 0; i < kMaxTopK; ++i) {
            if (i < topk) {
                ids[static_cast<size_t>(t) * topk + i] = id[i];
                weights[static_cast<size_t>(t) * topk + i] = z[i] / zs;
            }
        }
    }
    // Group counts and ranks: one ballot per expert over the group's tokens
    // (a token picks an expert at most once).
    const unsigned lt = (1u << lane) - 1u;
    for (int e = 0; e < experts; ++e) {
        int slot = -1;
#pragma unroll
        for (int i = 0; i < kMaxTopK; ++i)
            if (live && i < topk && id[i] == e) slot = i;
        const unsigned mask = __ballot_sync(0xFFFFFFFFu, slot >= 0);
        if (lane == 0) grp_count[static_cast<size_t>(group) * experts + e] = __popc(mask);
        if (slot >= 0) rank[static_cast<size_t>(t) * topk + slot] = __popc(mask & lt);
    }
}

// One CTA, thread e per expert (loops if experts > blockDim).  Replaces the
// group counts by each group's first sorted row for that expert.
__global__ void __launch_bounds__(1024)
    route_scan_kernel(int groups, int experts, int32_t* __restrict__ grp, int32_t* __restrict__ offsets) {
    __shared__ int warp_sum[32];
    const int e = threadIdx.x;
    int total = 0;
    if (e < experts)
        for (int g = 0; g < groups; ++g) total += grp[static_cast<size_t>(g) * experts + e];
    // Block-wide exclusive scan of tot over experts.
    const int lane = e & 31, w = e >> 5;
    int incl = total;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += y;
    }
    if (lane == 31) warp_sum[w] = incl;
    __syncthreads();
    if (w == 0) {
        int s = lane < (blockDim.x >> 5) ? warp_sum[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, s, d);
            if (lane >= d) s += y;
        }
        warp_sum[lane] = s;  // inclusive over warps
    }
    __syncthreads();
    const int base = incl - total + (w > 0 ? warp_sum[w - 1] : 0);
    if (e < experts) {
        offsets[e] = base;
        int run = base;
        for (int g = 0; g < groups; ++g) {
            const size_t i = static_cast<size_t>(g) * experts + e;
            const int c = grp[i];
            grp[i] = run;
            run += c;
        }
    }
    if (e == experts - 1) offsets[experts] = base + total;
}

__global__ void route_assign_kernel(int tokens, int experts, int topk, const int32_t* __restrict__ ids,
                                    const int32_t* __restrict__ grp, const int32_t* __restrict__ rank,
                                    int32_t* __restrict__ row_of, int32_t* __restrict__ sorted_token) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<int64_t>(tokens) * topk) return;
    const int t = static_cast<int>(i / topk);
    const int e = ids[i];
    const int r = grp[static_cast<size_t>(t >> 5) * experts + e] + rank[i];
    row_of[i] = r;
    sorted_token[r] = t;
}

// One warp per (token, 256-column chunk): lane c8 sums 8 columns over the
// token's k rows in slot order.
constexpr int kFinThreads = 256;
__global__ void __launch_bounds__(kFinThreads)
    finalize_kernel(const __nv_bfloat16* __restrict__ y2, const int32_t* __restrict__ row_of,
                    const float* __restrict__ weights, int64_t tokens, int topk, int64_t hidden,
                    __nv_bfloat16* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t chunks = (hidden + 255) >> 8;
    const int64_t total = tokens * chunks;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kFinThreads) >> 5;
    for (int64_t wi = (static_cast<int64_t>(blockIdx.x) * kFinThreads + threadIdx.x) >> 5; wi < total;
         wi += nwarps) {
        const int64_t t = wi / chunks;
        const int64_t c0 = (wi - t * chunks) * 256 + lane * 8;
        if (c0 >= hidden) continue;
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int s = 0; s < topk; ++s) {
            const int64_t r = row_of[t * topk + s];
            const float w = weights[t * topk + s];
            const uint4 raw = *reinterpret_cast<const uint4*>(y2 + r * hidden + c0);
            const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] += w * __uint_as_float(wd[i] << 16);
                acc[2 * i + 1] += w * __uint_as_float(wd[i] & 0xFFFF0000u);
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i]));
            const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i + 1]));
            o[i] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4*>(out + t * hidden + c0) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

cudaError_t launch_moe_route(const float* logits, int64_t tokens, int64_t experts, int64_t topk, int method,
                             int32_t* ids, float* weights, int32_t* offsets, int32_t* sorted_token,
                             int32_t* row_of, int32_t* ws, cudaStream_t s) {
    const int groups = static_cast<int>((tokens + 31) / 32);
    int32_t* grp = ws;
    int32_t* rank = ws + static_cast<size_t>(groups) * experts;
    const int blocks = (groups * 32 + kRouteThreads - 1) / kRouteThreads;
    route_topk_kernel<<<blocks, kRouteThreads, 0, s>>>(logits, static_cast<int>(tokens), static_cast<int>(experts),
                                                       static_cast<int>(topk), method, ids, weights, grp, rank);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    route_scan_kernel<<<1, 1024, 0, s>>>(groups, static_cast<int>(experts), grp, offsets);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t pairs = tokens * topk;
    route_assign_kernel<<<static_cast<int>((pairs + 255) / 256), 256, 0, s>>>(
        static_cast<int>(tokens), static_cast<int>(experts), static_cast<int>(topk), ids, grp, rank, row_of,
        sorted_token);
    return cudaGetLastError();
}

cudaError_t launch_moe_finalize(const void* y2, const int32_t* row_of, const float* weights, int64_t tokens,
                                int64_t topk, int64_t hidden, void* out, int num_sms, cudaStream_t s) {
    const int64_t work = tokens * ((hidden + 255) / 256);  // warps of work
    int64_t blocks = (work + (kFinThreads / 32) - 1) / (kFinThreads / 32);
    if (blocks > static_cast<int64_t>(num_sms) * 8) blocks = static_cast<int64_t>(num_sms) * 8;
    if (blocks < 1) blocks = 1;
    finalize_kernel<<<static_cast<int>(blocks), kFinThreads, 0, s>>>(
        static_cast<const __nv_bfloat16*>(y2), row_of, weights, tokens, static_cast<int>(topk), hidden,
        static_cast<__nv_bfloat16*>(out));
    return cudaGetLastError();
}

}  // namespace mxk
