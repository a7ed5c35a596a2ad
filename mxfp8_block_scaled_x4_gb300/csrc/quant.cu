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
// Work unit: one warp quantizes one 256-element chunk of one row (eight
// 32-blocks, four lanes per block, one 16-byte BF16 load per lane) -- fully
// coalesced 512-byte reads and 256-byte E4M3 writes per warp.  The four scale
// bytes of a 4-block group form one aligned 32-bit word in both scale layouts,
// so each half-warp writes one word.  Both kernels are HBM-bound: grids are
// sized to the SM count and each warp keeps UNROLL chunks in flight.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant_block.cuh"

namespace mxk {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

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

// Activations: rows [0, m8) x chunks of 256.  Rows >= m only write their
// (zero) scale words, which is what the 8x4 layout holds for padding rows.
__global__ void __launch_bounds__(kThreads) quant_act_kernel(const __nv_bfloat16* __restrict__ x,
                                                             int64_t m, int64_t m8, int64_t k,
                                                             uint8_t* __restrict__ q,
                                                             uint8_t* __restrict__ sf) {
    // Dependent kernels (the GEMM) may start their prologue now; they wait
    // for this grid's completion before reading what it writes.
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t chunks = k >> 8;
    const int64_t total = m8 * chunks;
    const int64_t kq = k >> 7;  // 4-block groups per row
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
    int64_t t0 = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    for (; t0 < total; t0 += nwarps * kUnroll) {
        uint4 raw[kUnroll];
        int64_t row[kUnroll], chunk[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t t = t0 + u * nwarps;
            row[u] = t / chunks;
            chunk[u] = t - row[u] * chunks;
            raw[u] = make_uint4(0, 0, 0, 0);
            if (t < total && row[u] < m)
                raw[u] = ld_nc_v4(x + row[u] * k + chunk[u] * 256 + lane * 8);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t t = t0 + u * nwarps;
            if (t >= total) break;  // warp-uniform
            float v[8];
            bf16x8_to_float(raw[u], v);
            uint2 qq;
            uint32_t s;
            quantize_lane8(v, qq, s);
            const uint32_t word = gather_scale_word(s);
            const int64_t r = row[u];
            if (r < m) st_v2(q + r * k + chunk[u] * 256 + lane * 8, qq);
            if ((lane & 15) == 0) {
                const int64_t grp = chunk[u] * 2 + (lane >> 4);
                *reinterpret_cast<uint32_t*>(sf + ((r >> 3) * kq + grp) * 32 + (r & 7) * 4) = word;
            }
        }
    }
}

// Weights: experts x rows [0, n_pad) x chunks.  Rows >= n write zero data and
// zero scales.  Scale word of (row r, 4-block group g) in the prepared layout:
// tile (r/128, g) of 512 bytes, inner offset (r%32)*16 + ((r%128)/32)*4.
template <bool kBf16>
__global__ void __launch_bounds__(kThreads)
    prepare_weight_kernel(const void* __restrict__ src, int64_t experts, int64_t n, int64_t n_pad,
                          int64_t k, uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
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
            const int64_t off = (e * n + r) * k + chunk * 256 + lane * 8;
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
        st_v2(q + rowp * k + chunk * 256 + lane * 8, qq);  // zero bytes for padding rows
        if ((lane & 15) == 0) {
            const int64_t grp = chunk * 2 + (lane >> 4);
            const int64_t tile = e * (n_pad >> 7) + (r >> 7);
            const int64_t rr = r & 127;
            *reinterpret_cast<uint32_t*>(sf + (tile * kq + grp) * 512 + (rr & 31) * 16 +
                                         (rr >> 5) * 4) = word;
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

cudaError_t launch_quant_act(const void* x, int64_t m, int64_t k, uint8_t* q, uint8_t* sf,
                             int num_sms, cudaStream_t s) {
    const int64_t m8 = (m + 7) / 8 * 8;
    const int64_t work = m8 * (k / 256);
    quant_act_kernel<<<grid_for(work, num_sms, kUnroll), kThreads, 0, s>>>(
        static_cast<const __nv_bfloat16*>(x), m, m8, k, q, sf);
    return cudaGetLastError();
}

cudaError_t launch_prepare_weight(const void* src, bool src_is_bf16, int64_t experts, int64_t n,
                                  int64_t n_pad, int64_t k, uint8_t* q, uint8_t* sf, int num_sms,
                                  cudaStream_t s) {
    const int64_t work = experts * n_pad * (k / 256);
    const int grid = grid_for(work, num_sms, 2);
    if (src_is_bf16)
        prepare_weight_kernel<true><<<grid, kThreads, 0, s>>>(src, experts, n, n_pad, k, q, sf);
    else
        prepare_weight_kernel<false><<<grid, kThreads, 0, s>>>(src, experts, n, n_pad, k, q, sf);
    return cudaGetLastError();
}

}  // namespace mxk
