// moe.cu -- routing and finalize kernels of the MXFP8 mixture-of-experts
// expert MLP.
//
// Routing follows FlashInfer PR #1214 "TRT-LLM Gen MoE" (Highlights): the
// Renormalize method (top-k of the logits, then a softmax over those k) and
// RenormalizeNaive (a softmax over all experts, top-k, then the k picks
// rescaled to sum to 1).  The experts of a token are chosen on the raw
// logits (the softmax is strictly monotone, so this is the top-k of the
// probabilities in exact arithmetic), in descending order, ties to the lower
// expert id.  The (token, slot) pairs are then sorted by expert, then token
// -- stable and deterministic, no order-dependent atomics:
//   route_cluster_kernel  up to kClusterTokens tokens, one launch: a cluster
//                       of 8 CTAs, one warp per token; per 32-token group a
//                       mask of the group's tokens per expert; the groups'
//                       counts exchanged through distributed shared memory
//                       -> offsets, then row_of[t*k + s] and
//                       sorted_token[row];
//   route_topk_kernel   above that, one CTA per 8-token group, one warp per
//                       token: the same selection and weights, then
//                       per-expert token masks -> group counts and each
//                       pair's rank inside its group;
//   route_scan_assign_kernel  one CTA: per-expert totals -> offsets, per
//                       (group, expert) the first sorted row of that group,
//                       then row_of[t*k + s] and sorted_token[row].
// Inside the layer, scatter_quant_kernel then quantizes each token's row of x
// once and writes it to the token's k expert-sorted rows (GEMM1's
// activations).  Finalize sums each token's k expert outputs with its
// routing weights in slot order (FP32) and rounds once to BF16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>

#include "internal.h"
#include "debug_check.cuh"
#include "ptx.cuh"
#include "quant_block.cuh"

namespace mxk {

namespace {

constexpr int kMaxTopK = 16;
constexpr int kMaxExpertsRoute = 1024;
// Tokens per routing group (one CTA of route_topk_kernel, one warp per
// token): small groups spread the selections over many SMs.
constexpr int kGroup = 8;
// Largest group-count table route_scan_assign_kernel stages in shared memory
// (48 KB less its own 128-byte static block).
constexpr size_t kScanSmemBytes = 48 * 1024 - 128;

// (v, e) ranks above (bv, be): larger logit, or equal logit and lower id.
__device__ __forceinline__ bool better(float v, int e, float bv, int be) {
    return v > bv || (v == bv && e < be);
}

// Logits of one token held by its warp: lane l keeps experts l, l + 32, ...
// (up to kRegLogits per lane, i.e. 256 experts) in registers so that the k
// selection rounds do not reload them; wider layers read them each round.
constexpr int kRegLogits = 8;

struct TokenLogits {
    float v[kRegLogits];
};

__device__ __forceinline__ void load_token_logits(const float* __restrict__ lg, int experts, int lane,
                                                  TokenLogits& tl) {
#pragma unroll
    for (int i = 0; i < kRegLogits; ++i) {
        const int e = lane + 32 * i;
        tl.v[i] = e < experts ? lg[e] : -INFINITY;
    }
}

// Order-preserving integer key of a logit: a larger key is a larger value;
// -0 and +0 share one key (they compare equal) and NaN takes the lowest key.
__device__ __forceinline__ uint32_t logit_key(float v) {
    if (v != v) return 0u;
    if (v == 0.0f) v = 0.0f;
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Sum over the warp (fixed butterfly: every lane gets the same value).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, d);
    return v;
}

// Inverse of logit_key (the shared key of +-0 reads back as +0, which
// changes no weight: only differences with the largest pick are used).
__device__ __forceinline__ float key_logit(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Selection with the logits in registers, NREG per lane (lane l holds experts
// l, l + 32, ...): every round each lane offers its best untaken key, the warp
// takes the largest (redux.sync max) and, among the lanes holding it, the
// lowest expert id (redux.sync min); the owning lane marks it taken.  Lane r
// keeps pick r.  Keys are computed once; the rounds are a loop, not unrolled
// (the kernel runs once per layer on SMs whose instruction cache is cold).
template <int NREG>
__device__ __forceinline__ void select_in_regs(const TokenLogits& tl, int experts, int topk, int lane, float& my_v,
                                               int& my_e, float& top0) {
    uint32_t key[NREG];
    uint32_t avail = 0u;  // bit i: logit i of this lane exists and is not yet taken
#pragma unroll
    for (int i = 0; i < NREG; ++i) {
        key[i] = logit_key(tl.v[i]);
        if (lane + 32 * i < experts) avail |= 1u << i;
    }
#pragma unroll 1
    for (int r = 0; r < topk; ++r) {
        uint32_t lk = 0u;
        int li = -1;
#pragma unroll
        for (int i = 0; i < NREG; ++i)
            if (((avail >> i) & 1u) && (li < 0 || key[i] > lk)) { lk = key[i]; li = i; }
        const uint32_t wk = __reduce_max_sync(0xFFFFFFFFu, li >= 0 ? lk : 0u);
        const uint32_t cand = (li >= 0 && lk == wk) ? static_cast<uint32_t>(lane + 32 * li) : 0xFFFFFFFFu;
        const int be = static_cast<int>(__reduce_min_sync(0xFFFFFFFFu, cand));
        if ((be & 31) == lane) avail &= ~(1u << (be >> 5));
        const float bv = key_logit(wk);
        if (lane == r) { my_v = bv; my_e = be; }
        if (r == 0) top0 = bv;
    }
}

// Top-k of one token by its warp and its weights.  Round r picks the best
// logit not yet taken (larger value, then lower id), so the picks come out in
// that total order; lane r keeps pick r.  Logits in registers (experts <=
// 32 * kRegLogits) go through select_in_regs; wider layers rescan the logits
// each round (lane-strided scan + butterfly arg-max, excluding earlier picks
// by order).  Lane r < topk writes id r (global, and sel_row if given) and
// weight r.
__device__ __forceinline__ void route_token(const float* __restrict__ lg, const TokenLogits& tl, int experts,
                                            int topk, int method, int lane, int32_t* __restrict__ ids_t,
                                            float* __restrict__ w_t, int* sel_row, int64_t base, int64_t extent) {
    const bool in_regs = experts <= 32 * kRegLogits;
    float my_v = 0.0f, top0 = 0.0f;
    int my_e = 0;
    if (experts <= 32 * 4) {
        select_in_regs<4>(tl, experts, topk, lane, my_v, my_e, top0);
    } else if (in_regs) {
        select_in_regs<kRegLogits>(tl, experts, topk, lane, my_v, my_e, top0);
    } else {
        float pv = INFINITY;
        int pe = -1;  // previous pick; round 0 admits everything
#pragma unroll 1
        for (int r = 0; r < topk; ++r) {
            float bv = -INFINITY;
            int be = 0x7FFFFFFF;
            for (int e = lane; e < experts; e += 32) {
                const float v = lg[e];
                if (better(pv, pe, v, e) && better(v, e, bv, be)) { bv = v; be = e; }
            }
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) {
                const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, d);
                const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, d);
                if (better(ov, oe, bv, be)) { bv = ov; be = oe; }
            }
            if (lane == r) { my_v = bv; my_e = be; }
            if (r == 0) top0 = bv;
            pv = bv;
            pe = be;
        }
    }
    if (lane < topk) {
        if (store_ok(base + lane, 1, extent)) ids_t[lane] = my_e;  // ids_t = ids + base
        if (sel_row) sel_row[lane] = my_e;
    }
    // Weights (top0 is the token's largest logit).
    float z = lane < topk ? expf(my_v - top0) : 0.0f;
    if (method == 1) {
        // Softmax over all logits (lane-strided partial sums, then a fixed
        // butterfly: deterministic), then renormalize the k picks.
        float all = 0.0f;
        if (in_regs) {
#pragma unroll
            for (int i = 0; i < kRegLogits; ++i)
                if (lane + 32 * i < experts) all += expf(tl.v[i] - top0);
        } else {
            for (int e = lane; e < experts; e += 32) all += expf(lg[e] - top0);
        }
        z = z / warp_sum(all);
    }
    const float zs = warp_sum(z);
    if (lane < topk && store_ok(base + lane, 1, extent)) w_t[lane] = z / zs;
}

// One CTA per group of kGroup tokens, one warp per token.  The group's picks
// then go into per-expert token masks in shared memory (atomicOr: the result
// does not depend on the order), which give the group count of every expert
// and each pair's rank among the group's tokens.
__global__ void __launch_bounds__(32 * kGroup)
    route_topk_kernel(const float* __restrict__ logits, int tokens, int experts, int topk, int method,
                      int32_t* __restrict__ ids, float* __restrict__ weights,
                      int32_t* __restrict__ grp_count, int32_t* __restrict__ rank) {
    __shared__ int sel[kGroup][kMaxTopK];
    __shared__ unsigned bits[kMaxExpertsRoute];
    // Its one dependent, route_scan_assign_kernel, may start at once (it waits
    // for this grid before reading anything); this grid itself waits for the
    // kernel that produced the logits.
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const int group = blockIdx.x;
    const int t = group * kGroup + w;
    for (int e = threadIdx.x; e < experts; e += blockDim.x) bits[e] = 0u;
    if (t < tokens) {
        const float* lg = logits + static_cast<size_t>(t) * experts;
        TokenLogits tl;
        if (experts <= 32 * kRegLogits) load_token_logits(lg, experts, lane, tl);
        route_token(lg, tl, experts, topk, method, lane, ids + static_cast<size_t>(t) * topk,
                    weights + static_cast<size_t>(t) * topk, sel[w], static_cast<int64_t>(t) * topk,
                    static_cast<int64_t>(tokens) * topk);
    }
    __syncthreads();
    const int live = min(kGroup, tokens - group * kGroup);
    for (int i = threadIdx.x; i < live * topk; i += blockDim.x) atomicOr(&bits[sel[i / topk][i % topk]], 1u << (i / topk));
    __syncthreads();
    const int64_t pairs = static_cast<int64_t>(tokens) * topk;
    const int64_t groups = (tokens + kGroup - 1) / kGroup;
    for (int i = threadIdx.x; i < live * topk; i += blockDim.x) {
        const int tw = i / topk;
        const int64_t o = static_cast<int64_t>(group * kGroup + tw) * topk + (i % topk);
        if (store_ok(o, 1, pairs)) rank[o] = __popc(bits[sel[tw][i % topk]] & ((1u << tw) - 1u));
    }
    for (int e = threadIdx.x; e < experts; e += blockDim.x)
        if (store_ok(static_cast<int64_t>(group) * experts + e, 1, groups * experts))
            grp_count[static_cast<size_t>(group) * experts + e] = __popc(bits[e]);
}

// Exclusive prefix sum of v over the threads of the block in thread order
// (every thread calls it; warp_sum holds 32 ints of shared memory).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sum) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += y;
    }
    if (lane == 31) warp_sum[w] = incl;
    __syncthreads();
    if (w == 0) {
        int sw = lane < static_cast<int>(blockDim.x >> 5) ? warp_sum[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, sw, d);
            if (lane >= d) sw += y;
        }
        warp_sum[lane] = sw;  // inclusive over warps
    }
    __syncthreads();
    return incl - v + (w > 0 ? warp_sum[w - 1] : 0);
}

// One CTA (thread e per expert, experts <= 1024): per-expert totals over the
// groups -> offsets (block scan); each group's counts are replaced by the
// group's first sorted row for that expert; then every pair gets its row
// (group base + rank in the group) and each row its token.  When the group
// counts fit (use_smem) they are read once into shared memory with
// independent loads and every later step works there.
__global__ void __launch_bounds__(1024)
    route_scan_assign_kernel(int tokens, int experts, int topk, const int32_t* __restrict__ ids,
                             int32_t* __restrict__ grp, const int32_t* __restrict__ rank,
                             int32_t* __restrict__ offsets, int32_t* __restrict__ row_of,
                             int32_t* __restrict__ sorted_token, int use_smem, int release) {
    extern __shared__ int sgrp[];
    __shared__ int warp_sum[32];
    // Waits for route_topk_kernel.  Releases its dependent early only when
    // told, and only after that wait (inside the MoE layer: the scattering
    // quantizer, which reads x before its own wait and waits for this grid
    // before releasing the grouped GEMM that reads the offsets).
    pdl_wait();
    if (release) pdl_launch_dependents();
    const int groups = (tokens + kGroup - 1) / kGroup;
    const int64_t cells = static_cast<int64_t>(groups) * experts;
    int32_t* cnt = grp;
    if (use_smem) {
#pragma unroll 4
        for (int i = threadIdx.x; i < static_cast<int>(cells); i += blockDim.x) sgrp[i] = grp[i];
        __syncthreads();
        cnt = sgrp;
    }
    const int e = threadIdx.x;
    int total = 0;
    if (e < experts) {
#pragma unroll 8
        for (int g = 0; g < groups; ++g) total += cnt[static_cast<size_t>(g) * experts + e];
    }
    const int base = block_exclusive_scan(total, warp_sum);
    if (e < experts) {
        if (store_ok(e, 1, experts + 1)) offsets[e] = base;
        int run = base;
#pragma unroll 8
        for (int g = 0; g < groups; ++g) {
            const size_t i = static_cast<size_t>(g) * experts + e;
            const int c = cnt[i];
            if (use_smem || store_ok(static_cast<int64_t>(i), 1, cells)) cnt[i] = run;
            run += c;
        }
    }
    if (e == experts - 1) offsets[experts] = base + total;
    __syncthreads();  // this CTA's bases are visible to all of its threads
    const int pairs = tokens * topk;
#pragma unroll 2
    for (int i = threadIdx.x; i < pairs; i += blockDim.x) {
        const int t = i / topk;
        const int r = cnt[static_cast<size_t>(t / kGroup) * experts + ids[i]] + rank[i];
        if (store_ok(i, 1, pairs)) row_of[i] = r;
        if (store_ok(r, 1, pairs)) sorted_token[r] = t;
    }
}

// Routing in one launch for up to kClusterTokens tokens: one cluster of CTAS
// CTAs of WARPS warps (16 x 16 where the GPU schedules a 16-CTA cluster and
// experts <= 512: fewer tokens per SM; else 8 x 32).  Tokens form WARPS-token
// groups; group g is routed by CTA g % CTAS in pass g / CTAS, one warp per
// token.  Each CTA records, per pass and expert, the mask of the group's
// tokens that picked the expert.  After a cluster barrier every CTA reads
// all groups' counts (mask popcounts) from its peers' shared memory in group
// order, so that thread e knows expert e's total and the count before each of
// its own groups; a block scan of the totals gives the offsets (written by
// CTA 0), and each pair's row is its expert's offset + the count of earlier
// groups + its rank among the group's tokens (a popcount of the mask below
// it): the stable expert-sorted order.  A second barrier phase keeps every
// CTA alive until no peer reads its masks any more.  The kernel releases its
// dependent early only when told (`release`), and only after its own
// dependency wait: inside the MoE layer, whose next kernel is the scattering
// quantizer (it reads x before its wait, and waits for this grid before it
// releases the grouped GEMM, which reads the offsets in its prologue).
constexpr int kClusterMaxPasses = 2;
constexpr int kClusterTokens = 512;  // CTAS * WARPS * kClusterMaxPasses for both shapes below
template <int CTAS, int WARPS>
__global__ void __launch_bounds__(32 * WARPS, 1)
    route_cluster_kernel(const float* __restrict__ logits, int tokens, int experts, int topk, int method,
                         int32_t* __restrict__ ids, float* __restrict__ weights, int32_t* __restrict__ offsets,
                         int32_t* __restrict__ row_of, int32_t* __restrict__ sorted_token, int release) {
    extern __shared__ uint32_t route_smem[];  // masks [passes][experts], then bases [passes][experts]
    __shared__ int sel[kClusterMaxPasses][WARPS][kMaxTopK];
    __shared__ int warp_sum[32];
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const int crank = static_cast<int>(cluster_rank());
    const int groups = (tokens + WARPS - 1) / WARPS;
    const int passes = (groups + CTAS - 1) / CTAS;
    uint32_t* masks = route_smem;
    int* base = reinterpret_cast<int*>(route_smem + passes * experts);
    for (int i = threadIdx.x; i < passes * experts; i += blockDim.x) masks[i] = 0u;
    pdl_wait();  // the logits come from the previous kernel
    if (release) pdl_launch_dependents();
    const int64_t pairs = static_cast<int64_t>(tokens) * topk;
    for (int j = 0; j < passes; ++j) {
        const int t = (j * CTAS + crank) * WARPS + w;
        if (t < tokens) {
            const float* lg = logits + static_cast<size_t>(t) * experts;
            TokenLogits tl;
            if (experts <= 32 * kRegLogits) load_token_logits(lg, experts, lane, tl);
            route_token(lg, tl, experts, topk, method, lane, ids + static_cast<size_t>(t) * topk,
                        weights + static_cast<size_t>(t) * topk, sel[j][w], static_cast<int64_t>(t) * topk, pairs);
        }
    }
    __syncthreads();
    const int local_pairs = passes * WARPS * topk;
    for (int i = threadIdx.x; i < local_pairs; i += blockDim.x) {
        const int j = i / (WARPS * topk), tw = (i / topk) % WARPS;
        if ((j * CTAS + crank) * WARPS + tw < tokens) atomicOr(&masks[j * experts + sel[j][tw][i % topk]], 1u << tw);
    }
    cluster_arrive_release();  // every CTA's masks are complete ...
    cluster_wait_acquire();    // ... before any peer reads them
    const int e = threadIdx.x;
    int total = 0;
    int before[kClusterMaxPasses];
#pragma unroll
    for (int j = 0; j < kClusterMaxPasses; ++j) before[j] = 0;
    if (e < experts) {
        // All of a chunk's remote loads go out before any is used: one
        // DSMEM round trip per chunk instead of one per few groups.
        constexpr int kChunk = 16;
        for (int g0 = 0; g0 < groups; g0 += kChunk) {
            uint32_t mk[kChunk];
#pragma unroll
            for (int k = 0; k < kChunk; ++k) {
                const int g = g0 + k;
                mk[k] = g < groups ? ld_shared_cluster_u32(map_to_rank(smem_addr(&masks[(g / CTAS) * experts + e]),
                                                                       static_cast<uint32_t>(g % CTAS)))
                                   : 0u;
            }
#pragma unroll
            for (int k = 0; k < kChunk; ++k) {
                const int g = g0 + k;
                const int c = __popc(mk[k]);
#pragma unroll
                for (int j = 0; j < kClusterMaxPasses; ++j)
                    if (g < j * CTAS + crank) before[j] += c;
                total += c;
            }
        }
    }
    cluster_arrive_relaxed();  // this thread's remote reads are done
    const int off = block_exclusive_scan(e < experts ? total : 0, warp_sum);
    if (e < experts) {
        if (crank == 0 && store_ok(e, 1, experts + 1)) offsets[e] = off;
        if (crank == 0 && e == experts - 1) offsets[experts] = off + total;
#pragma unroll
        for (int j = 0; j < kClusterMaxPasses; ++j)
            if (j < passes) base[j * experts + e] = off + before[j];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < local_pairs; i += blockDim.x) {
        const int j = i / (WARPS * topk), tw = (i / topk) % WARPS, sl = i % topk;
        const int t = (j * CTAS + crank) * WARPS + tw;
        if (t >= tokens) continue;
        const int ex = sel[j][tw][sl];
        const int r = base[j * experts + ex] + __popc(masks[j * experts + ex] & ((1u << tw) - 1u));
        const int64_t pi = static_cast<int64_t>(t) * topk + sl;
        if (store_ok(pi, 1, pairs)) row_of[pi] = r;
        if (store_ok(r, 1, pairs)) sorted_token[r] = t;
    }
    cluster_wait();  // no peer reads this CTA's masks any more
}

// GEMM1's activation rows in the MoE layer, by token: lane (t, b) quantizes
// 32-block b of token t's row of x once (the activation quantizer's
// arithmetic: E4M3 bytes and one E8M0 scale per block) and writes it to the
// token's topk expert-sorted rows row_of[t * topk + s] of qa, the scale
// bytes in the 8x4 layout; block 0 then gives rows pairs .. ceil8(pairs)-1
// of the last scale group zero scales, as the quantizer does.  Nothing before
// the dependency wait depends on the routing: each lane's first block is
// loaded and quantized while the router runs (x is complete by then: the
// router releases this grid only after its own wait); row_of is read after
// the wait.  The grouped GEMM is released after the wait too (it reads the
// expert offsets in its prologue).  Thin CTAs (at most 64 registers a
// thread) so that GEMM1's CTA fits beside one on an SM.
constexpr int kScatThreads = 128;
__global__ void __launch_bounds__(kScatThreads, 8)
    scatter_quant_kernel(const __nv_bfloat16* __restrict__ x, int64_t tokens, int topk, int64_t k,
                         const int32_t* __restrict__ row_of, uint8_t* __restrict__ qa, uint8_t* __restrict__ sfa) {
    const int64_t kb = k >> 5;  // 32-blocks per row (a multiple of 4)
    const int64_t total = tokens * kb;
    const int64_t pairs = tokens * topk;
    const int64_t rows8 = (pairs + 7) & ~static_cast<int64_t>(7);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kScatThreads;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * kScatThreads + threadIdx.x;
    // Task t * kb + b starts at x + (t * kb + b) * 32.
    auto quantize = [&](int64_t task, uint32_t (&qq)[8]) {
        const uint4* src = reinterpret_cast<const uint4*>(x + task * 32);
        const uint4 raw[4] = {src[0], src[1], src[2], src[3]};
        return quantize_block32(raw, qq);
    };
    auto scatter = [&](int64_t task, const uint32_t (&qq)[8], uint32_t sc) {
        const int64_t t = task / kb, b = task - t * kb;
        int rows[kMaxTopK];
#pragma unroll
        for (int sl = 0; sl < kMaxTopK; ++sl) rows[sl] = sl < topk ? row_of[t * topk + sl] : 0;
#pragma unroll
        for (int sl = 0; sl < kMaxTopK; ++sl) {
            if (sl >= topk) break;
            const int64_t r = rows[sl];
            if (store_ok(r * k + b * 32, 32, pairs * k)) {
                uint4* dst = reinterpret_cast<uint4*>(qa + r * k + b * 32);
                dst[0] = make_uint4(qq[0], qq[1], qq[2], qq[3]);
                dst[1] = make_uint4(qq[4], qq[5], qq[6], qq[7]);
            }
            const int64_t o = ((r >> 3) * (kb >> 2) + (b >> 2)) * 32 + (r & 7) * 4 + (b & 3);
            if (store_ok(o, 1, rows8 * kb)) sfa[o] = static_cast<uint8_t>(sc);
        }
    };
    uint32_t q0[8];
    uint32_t s0 = 0;
    if (first < total) s0 = quantize(first, q0);
    pdl_wait();  // row_of comes from the router
    pdl_launch_dependents();
    if (first < total) scatter(first, q0, s0);
    for (int64_t task = first + stride; task < total; task += stride) {
        uint32_t qq[8];
        const uint32_t sc = quantize(task, qq);
        scatter(task, qq, sc);
    }
    if (blockIdx.x == 0) {
        for (int64_t i = threadIdx.x; i < (rows8 - pairs) * kb; i += kScatThreads) {
            const int64_t r = pairs + i / kb, b = i % kb;
            const int64_t o = ((r >> 3) * (kb >> 2) + (b >> 2)) * 32 + (r & 7) * 4 + (b & 3);
            if (store_ok(o, 1, rows8 * kb)) sfa[o] = 0;
        }
    }
}

// One warp per (token, 256-column chunk): lane c8 sums 8 columns over the
// token's k rows in slot order.  Slots go in chunks of kFinChunk: the
// chunk's row indices and weights are loaded first, then its row segments,
// so the loads overlap instead of forming k dependent round trips; the sum
// keeps slot order.  Four-warp CTAs with a small register footprint stay
// resident beside the grouped GEMM before it, waiting for it to finish.
constexpr int kFinThreads = 128;
constexpr int kFinChunk = 8;
__global__ void __launch_bounds__(kFinThreads)
    finalize_kernel(const __nv_bfloat16* __restrict__ y2, const int32_t* __restrict__ row_of,
                    const float* __restrict__ weights, int64_t tokens, int topk, int64_t hidden,
                    __nv_bfloat16* __restrict__ out, int slots_ready) {
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t chunks = (hidden + 255) >> 8;
    const int64_t total = tokens * chunks;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kFinThreads) >> 5;
    const int64_t first = (static_cast<int64_t>(blockIdx.x) * kFinThreads + threadIdx.x) >> 5;
    int rows[kFinChunk];
    float wts[kFinChunk];
    auto load_slots = [&](int64_t t, int s0) {
#pragma unroll
        for (int j = 0; j < kFinChunk; ++j) {
            const bool live = s0 + j < topk;
            rows[j] = live ? row_of[t * topk + s0 + j] : 0;
            wts[j] = live ? weights[t * topk + s0 + j] : 0.0f;
        }
    };
    // slots_ready: row_of and the weights were complete before the kernel
    // this grid depends on began (inside the MoE layer they come from its
    // routing kernel), so the first item's slots load before the wait.
    const bool early = slots_ready && first < total;
    if (early) load_slots(first / chunks, 0);
    pdl_wait();  // y2 comes from the previous kernel
    for (int64_t wi = first; wi < total; wi += nwarps) {
        const int64_t t = wi / chunks;
        const int64_t c0 = (wi - t * chunks) * 256 + lane * 8;
        if (c0 >= hidden) continue;
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int s0 = 0; s0 < topk; s0 += kFinChunk) {
            if (!(early && wi == first && s0 == 0)) load_slots(t, s0);
            uint4 raw[kFinChunk];
#pragma unroll
            for (int j = 0; j < kFinChunk; ++j)
                raw[j] = s0 + j < topk
                             ? *reinterpret_cast<const uint4*>(y2 + static_cast<int64_t>(rows[j]) * hidden + c0)
                             : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int j = 0; j < kFinChunk; ++j) {
                if (s0 + j >= topk) break;
                const uint32_t wd[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] += wts[j] * __uint_as_float(wd[i] << 16);
                    acc[2 * i + 1] += wts[j] * __uint_as_float(wd[i] & 0xFFFF0000u);
                }
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i]));
            const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i + 1]));
            o[i] = lo | (hi << 16);
        }
        if (store_ok(t * hidden + c0, 8, tokens * hidden))
            *reinterpret_cast<uint4*>(out + t * hidden + c0) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

cudaError_t read_and_clear_oob_moe(unsigned int* out) { return read_and_clear_oob_word(out); }

namespace {
// Whether this GPU schedules the routing kernel as one 16-CTA cluster (a
// size beyond the portable 8, allowed per kernel); asked once per device.
bool cluster16_schedulable() {
    static std::atomic<int> cached[64];  // 0 unknown, 1 yes, -1 no
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    const int known = cached[dev].load(std::memory_order_relaxed);
    if (known != 0) return known > 0;
    bool ok = cudaFuncSetAttribute(route_cluster_kernel<16, 16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
              cudaSuccess;
    if (ok) {
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof(cfg));
        cfg.gridDim = dim3(16, 1, 1);
        cfg.blockDim = dim3(512, 1, 1);
        cfg.dynamicSmemBytes = 2 * 512 * 2 * sizeof(uint32_t);
        cudaLaunchAttribute a;
        a.id = cudaLaunchAttributeClusterDimension;
        a.val.clusterDim.x = 16;
        a.val.clusterDim.y = 1;
        a.val.clusterDim.z = 1;
        cfg.attrs = &a;
        cfg.numAttrs = 1;
        int n = 0;
        ok = cudaOccupancyMaxActiveClusters(&n, route_cluster_kernel<16, 16>, &cfg) == cudaSuccess && n >= 1;
    }
    if (!ok) (void)cudaGetLastError();  // the probe's own failure, not a caller's error
    cached[dev].store(ok ? 1 : -1, std::memory_order_relaxed);
    return ok;
}
}  // namespace

// The routing kernels are launched with programmatic stream serialization so
// that their launches overlap the kernel before them (each waits for it
// before reading its inputs).  Up to kClusterTokens tokens one cluster kernel
// does everything; above, route_topk_kernel releases its dependent (the
// second routing kernel) at once.  The kernel that writes the offsets
// releases its own dependent early only with `release` (the MoE layer, whose
// next kernel is the gathering quantizer): the grouped GEMMs read the expert
// offsets in their prologue, before their own griddepcontrol.wait, so no
// grouped GEMM may start before the offsets are complete.
cudaError_t launch_moe_route(const float* logits, int64_t tokens, int64_t experts, int64_t topk, int method,
                             int32_t* ids, float* weights, int32_t* offsets, int32_t* sorted_token,
                             int32_t* row_of, int32_t* ws, cudaStream_t s, bool release) {
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.blockDim = dim3(1024, 1, 1);
    cfg.stream = s;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const int T = static_cast<int>(tokens), E = static_cast<int>(experts), K = static_cast<int>(topk);
    if (tokens <= kClusterTokens) {
        // One launch: a single cluster routes every token and sorts the pairs.
        const bool wide = E <= 512 && cluster16_schedulable();
        if (wide || E <= 1024) {
            const int ctas = wide ? 16 : 8, warps = wide ? 16 : 32;
            cudaLaunchAttribute attrs[2];
            attrs[0] = attr;
            attrs[1].id = cudaLaunchAttributeClusterDimension;
            attrs[1].val.clusterDim.x = ctas;
            attrs[1].val.clusterDim.y = 1;
            attrs[1].val.clusterDim.z = 1;
            cfg.attrs = attrs;
            cfg.numAttrs = 2;
            cfg.gridDim = dim3(ctas, 1, 1);
            cfg.blockDim = dim3(32 * warps, 1, 1);
            const int passes = (T + warps * ctas - 1) / (warps * ctas);
            cfg.dynamicSmemBytes = static_cast<size_t>(passes) * E * 2 * sizeof(uint32_t);
            if (wide)
                return cudaLaunchKernelEx(&cfg, route_cluster_kernel<16, 16>, logits, T, E, K, method, ids, weights,
                                          offsets, row_of, sorted_token, release ? 1 : 0);
            return cudaLaunchKernelEx(&cfg, route_cluster_kernel<8, 32>, logits, T, E, K, method, ids, weights,
                                      offsets, row_of, sorted_token, release ? 1 : 0);
        }
    }
    const int groups = static_cast<int>((tokens + kGroup - 1) / kGroup);
    int32_t* grp = ws;
    int32_t* rank = ws + static_cast<size_t>(groups) * experts;
    cfg.gridDim = dim3(groups, 1, 1);
    cfg.blockDim = dim3(32 * kGroup, 1, 1);
    cudaError_t e = cudaLaunchKernelEx(&cfg, route_topk_kernel, logits, T, E, K, method, ids, weights, grp, rank);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(1024, 1, 1);  // one thread per expert
    // Group counts in shared memory when they fit the default 48 KB.
    const size_t cells_bytes = static_cast<size_t>(groups) * experts * sizeof(int32_t);
    const int use_smem = cells_bytes <= kScanSmemBytes ? 1 : 0;
    cfg.dynamicSmemBytes = use_smem ? cells_bytes : 0;
    return cudaLaunchKernelEx(&cfg, route_scan_assign_kernel, T, E, K, static_cast<const int32_t*>(ids), grp,
                              static_cast<const int32_t*>(rank), offsets, row_of, sorted_token, use_smem,
                              release ? 1 : 0);
}

cudaError_t launch_moe_scatter_quant(const void* x, int64_t tokens, int64_t topk, int64_t k, const int32_t* row_of,
                                     uint8_t* qa, uint8_t* sfa, int num_sms, cudaStream_t s) {
    // An SM changes its L1 / shared-memory split only while idle: ask for the
    // largest shared carveout (once per device) so that an SM running one of
    // these CTAs can take a grouped GEMM CTA.
    static std::atomic<int> carveout_set[64];
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64 &&
        carveout_set[dev].load(std::memory_order_relaxed) == 0) {
        if (cudaFuncSetAttribute(scatter_quant_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            (void)cudaGetLastError();  // a hint only
        carveout_set[dev].store(1, std::memory_order_relaxed);
    }
    const int64_t total = tokens * (k / 32);
    int64_t blocks = (total + kScatThreads - 1) / kScatThreads;
    if (blocks > static_cast<int64_t>(num_sms) * 4) blocks = static_cast<int64_t>(num_sms) * 4;
    if (blocks < 1) blocks = 1;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(kScatThreads, 1, 1);
    cfg.stream = s;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, scatter_quant_kernel, static_cast<const __nv_bfloat16*>(x), tokens,
                              static_cast<int>(topk), k, row_of, qa, sfa);
}

cudaError_t launch_moe_finalize(const void* y2, const int32_t* row_of, const float* weights, int64_t tokens,
                                int64_t topk, int64_t hidden, void* out, int num_sms, cudaStream_t s,
                                bool slots_ready) {
    const int64_t work = tokens * ((hidden + 255) / 256);  // warps of work
    int64_t blocks = (work + (kFinThreads / 32) - 1) / (kFinThreads / 32);
    if (blocks > static_cast<int64_t>(num_sms) * 8) blocks = static_cast<int64_t>(num_sms) * 8;
    if (blocks < 1) blocks = 1;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(kFinThreads, 1, 1);
    cfg.stream = s;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, finalize_kernel, static_cast<const __nv_bfloat16*>(y2), row_of, weights, tokens,
                              static_cast<int>(topk), hidden, static_cast<__nv_bfloat16*>(out),
                              slots_ready ? 1 : 0);
}

}  // namespace mxk
