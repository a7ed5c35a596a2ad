// quant.cu -- the two MXFP8 quantization kernels.
//
//  * quant_act_kernel: per-call BF16 activation quantizer with the 8x4 scale
//    layout (vLLM PR #52204 "[Kernel] Add FlashInfer TRTLLM MXFP8 linear
//    backend": apply_weights quantizes BF16 activations "with the 8x4 scale
//    layout"; the prhub summary's fake implementation sizes the scale buffer
//    ceil(m/8)*8 * ceil(k/32/4)*4 bytes).
//  * prepare_weight_kernel: load-time weight preparation (same PR,
//    process_weights_after_loading: quantize, pad N to a multiple of 128,
//    lay data and scales out for the GEMM).
//
// Work units: the activation kernel gives each lane a whole 32-block of an
// 8-row x 128-column patch (one 8x4 scale tile per warp); the weight kernel
// quantizes one 256-element chunk of a row per warp (four lanes per block,
// one 16-byte load per lane), and each half-warp writes one aligned 32-bit
// word of the prepared 128x4 scale layout.  Both kernels are HBM-bound: grids
// are sized to the SM count and each warp keeps several units in flight.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "internal.h"
#include "ptx.cuh"
#include "debug_check.cuh"
#include "quant_block.cuh"

namespace mxk {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 2;

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void st_v2(void* p, uint2 v) {
    asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// Activations.  One warp quantizes an 8-row x 128-column patch: lane l owns
// row l/4 of the patch and its 32-block l%4 (64 contiguous BF16 bytes), so
// the block's amax needs no shuffle, the lane writes its 32 E4M3 bytes as two
// 16-byte stores, and the patch's 32 scale bytes -- exactly one 8x4 tile, byte
// (row%8)*4 + block%4 = lane -- go out as one coalesced 32-byte store.  Rows in
// [m, m8) quantize zeros and write only their (zero) scales.
// With `src_rows`, output row r reads input row src_rows[r] (a gather, e.g.
// tokens into expert-sorted order).  With `layout128`, the scales go to the
// 128x4 layout of the prepared weights instead (tile (row/128, K block) of
// 512 bytes, byte (row%32)*16 + ((row%128)/32)*4 + block%4; rows up to
// m_pad = ceil128(m)), one byte per lane.
template <bool kGather, bool kLayout128>
__global__ void __launch_bounds__(kThreads) quant_act_kernel(const __nv_bfloat16* __restrict__ x,
                                                             int64_t m, int64_t m8, int64_t k,
                                                             const int32_t* __restrict__ src_rows,
                                                             uint8_t* __restrict__ q,
                                                             uint8_t* __restrict__ sf) {
    // Dependent kernels (the GEMM) may start their prologue early; they wait
    // for this grid's completion before reading what it writes.  This grid
    // itself may start before the kernel that produced x has finished: every
    // CTA waits for it before touching x, q or sf.  The gathering variant
    // (MoE GEMM1's rows) releases its dependent only after that wait: the
    // grouped GEMM reads the expert offsets in its prologue, and they come
    // from the routing kernel this grid waits for.
    if constexpr (!kGather) pdl_launch_dependents();
    pdl_wait();
    if constexpr (kGather) pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t quads = k >> 7;  // 128-column patches per row group
    const int64_t total = (m8 >> 3) * quads;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
    const int r8 = lane >> 2;
    const int b4 = lane & 3;
    for (int64_t t0 = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5; t0 < total;
         t0 += nwarps * kUnroll) {
        uint4 raw[kUnroll][4];
        int64_t row[kUnroll], col[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t t = t0 + u * nwarps;
            const int64_t g = t / quads;
            row[u] = g * 8 + r8;
            col[u] = (t - g * quads) * 128 + b4 * 32;
#pragma unroll
            for (int i = 0; i < 4; ++i) raw[u][i] = make_uint4(0, 0, 0, 0);
            if (t < total && row[u] < m) {
                const int64_t sr = kGather ? static_cast<int64_t>(src_rows[row[u]]) : row[u];
                const __nv_bfloat16* src = x + sr * k + col[u];
#pragma unroll
                for (int i = 0; i < 4; ++i) raw[u][i] = *reinterpret_cast<const uint4*>(src + i * 8);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t t = t0 + u * nwarps;
            if (t >= total) break;  // warp-uniform
            uint32_t qq[8];
            const uint32_t s = quantize_block32(raw[u], qq);
            if (row[u] < m && store_ok(row[u] * k + col[u], 32, m * k)) {
                uint4* dst = reinterpret_cast<uint4*>(q + row[u] * k + col[u]);
                dst[0] = make_uint4(qq[0], qq[1], qq[2], qq[3]);
                dst[1] = make_uint4(qq[4], qq[5], qq[6], qq[7]);
            }
            const int64_t sf_extent = m8 * (k >> 5);  // 8x4: ceil8(m) rows; 128x4: ceil128(m) rows
            if constexpr (!kLayout128) {
                if (store_ok(t * 32 + lane, 1, sf_extent))
                    sf[t * 32 + lane] = static_cast<uint8_t>(s);  // 8x4 tile (g, quad) = t
            } else {
                const int64_t g = t / quads;
                const int64_t r = row[u];
                const int64_t o = ((r >> 7) * quads + (t - g * quads)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + b4;
                if (store_ok(o, 1, sf_extent)) sf[o] = static_cast<uint8_t>(s);
            }
        }
    }
}

// Weights: experts x rows [0, n_pad) x chunks.  Rows >= n write zero data and
// zero scales.  With `inter` > 0 (gated GEMM1 weights [gate; up], n = 2 inter)
// prepared row r of 128-row tile j = r / 128 reads gate row 64 j + r % 128
// for r % 128 < 64, else up row inter + 64 j + r % 128 - 64 (gated-row
// reorder: one tile yields 64 features of silu(gate) * up).  Scale word of (row r, 4-block group g) in the prepared layout:
// tile (r/128, g) of 512 bytes, inner offset (r%32)*16 + ((r%128)/32)*4.
template <bool kBf16>
__global__ void __launch_bounds__(kThreads)
    prepare_weight_kernel(const void* __restrict__ src, int64_t experts, int64_t n, int64_t n_pad,
                          int64_t k, int64_t inter, uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
    const int lane = threadIdx.x & 31;
    const int64_t chunks = k >> 8;
    const int64_t kq = k >> 7;
    const int64_t total = experts * n_pad * chunks;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
    int64_t t = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    for (; t < total; t += nwarps) {
        const int64_t rowp = t / chunks;  // row in the padded [experts * n_pad] space
        const int64_t chunk = t - rowp * chunks;
        const int64_t e = rowp / n_pad;
        const int64_t r = rowp - e * n_pad;
        float v[8];
        if (r < n) {
            const int64_t o = r & 127;
            const int64_t sr = inter <= 0 ? r : (o < 64 ? (r >> 7) * 64 + o : inter + (r >> 7) * 64 + o - 64);
            const int64_t off = (e * n + sr) * k + chunk * 256 + lane * 8;
            if (kBf16) {
                bf16x8_to_float(ld_nc_v4(static_cast<const __nv_bfloat16*>(src) + off), v);
            } else {
                const float* f = static_cast<const float*>(src) + off;
                const uint4 a = ld_nc_v4(f);
                const uint4 b = ld_nc_v4(f + 4);
                v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
                v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
                v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
                v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.0f;
        }
        uint2 qq;
        uint32_t s;
        quantize_lane8(v, qq, s);
        const uint32_t word = gather_scale_word(s);
        if (store_ok(rowp * k + chunk * 256 + lane * 8, 8, experts * n_pad * k))
            st_v2(q + rowp * k + chunk * 256 + lane * 8, qq);  // zero bytes for padding rows
        if ((lane & 15) == 0) {
            const int64_t grp = chunk * 2 + (lane >> 4);
            const int64_t tile = e * (n_pad >> 7) + (r >> 7);
            const int64_t rr = r & 127;
            const int64_t o = (tile * kq + grp) * 512 + (rr & 31) * 16 + (rr >> 5) * 4;
            if (store_ok(o, 4, experts * n_pad * (k >> 5))) *reinterpret_cast<uint32_t*>(sf + o) = word;
        }
    }
}

int grid_for(int64_t warps_of_work, int num_sms, int per_warp) {
    const int64_t warps_per_block = kThreads / 32;
    int64_t blocks = (warps_of_work + warps_per_block * per_warp - 1) / (warps_per_block * per_warp);
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;  // 8 x 256 threads = full SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

}  // namespace

cudaError_t read_and_clear_oob_quant(unsigned int* out) { return read_and_clear_oob_word(out); }

cudaError_t launch_quant_act(const void* x, int64_t m, int64_t k, uint8_t* q, uint8_t* sf,
                             int num_sms, cudaStream_t s, const int32_t* src_rows, bool layout_128x4) {
    // Rows past m quantize zeros and write zero scales: up to ceil8(m) for
    // the 8x4 layout, ceil128(m) for the 128x4 one.
    const int64_t m8 = layout_128x4 ? (m + 127) / 128 * 128 : (m + 7) / 8 * 8;
    const int64_t work = (m8 / 8) * (k / 128);
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(grid_for(work, num_sms, kUnroll), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    if (src_rows && layout_128x4) return cudaErrorInvalidValue;
    if (src_rows) return cudaLaunchKernelEx(&cfg, quant_act_kernel<true, false>, xb, m, m8, k, src_rows, q, sf);
    if (layout_128x4) return cudaLaunchKernelEx(&cfg, quant_act_kernel<false, true>, xb, m, m8, k, src_rows, q, sf);
    return cudaLaunchKernelEx(&cfg, quant_act_kernel<false, false>, xb, m, m8, k, src_rows, q, sf);
}

cudaError_t launch_prepare_weight(const void* src, bool src_is_bf16, int64_t experts, int64_t n,
                                  int64_t n_pad, int64_t k, uint8_t* q, uint8_t* sf, int num_sms,
                                  cudaStream_t s, int64_t inter) {
    const int64_t work = experts * n_pad * (k / 256);
    const int grid = grid_for(work, num_sms, 2);
    if (src_is_bf16)
        prepare_weight_kernel<true><<<grid, kThreads, 0, s>>>(src, experts, n, n_pad, k, inter, q, sf);
    else
        prepare_weight_kernel<false><<<grid, kThreads, 0, s>>>(src, experts, n, n_pad, k, inter, q, sf);
    return cudaGetLastError();
}

}  // namespace mxk
