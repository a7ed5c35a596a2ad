// quant_block.cuh -- MXFP8 quantization of one 32-element block by four lanes.
//
// Four consecutive lanes (4i .. 4i+3) hold the 32 values of one block, eight
// each, widened exactly to float.  The block's amax is reduced with two
// butterfly shuffles on the magnitude bits (for finite non-negative floats the
// integer order of the bit patterns is the numeric order).  Scale rule (the
// OCP MX v1.0 rule for MXFP8, which the pages name as the format):
//   byte = clamp(floor(log2(amax)) - 8 + 127, 0, 254)
// computed from amax's biased exponent field E (floor(log2) = E - 127 for
// normal amax; subnormal and zero amax clamp to byte 0).  Elements are
// v * 2^(127 - byte), an exact power-of-two multiply, then converted with the
// hardware round-to-nearest-even, saturate-to-finite E4M3 conversion.  A block
// holding Inf or NaN gets byte 0xFF and elements 0x7F.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace mxk {

__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    __nv_fp8x2_storage_t r =
        __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
    return static_cast<uint32_t>(r);
}

// v: this lane's 8 values.  Must be called by all 32 lanes of the warp.
// Returns the 8 E4M3 bytes (little-endian in q) and this lane's block's
// scale byte.
__device__ __forceinline__ void quantize_lane8(const float (&v)[8], uint2& q, uint32_t& scale) {
    uint32_t a = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = max(a, __float_as_uint(v[i]) & 0x7FFFFFFFu);
    a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
    a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
    if (a >= 0x7F800000u) {  // Inf or NaN somewhere in the block
        scale = 0xFFu;
        q = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
        return;
    }
    int sb = static_cast<int>(a >> 23) - 8;  // floor(log2(amax)) - 8 + 127
    sb = sb < 0 ? 0 : sb;                    // never above 246 for finite amax
    const float mul = __uint_as_float(static_cast<uint32_t>(254 - sb) << 23);  // 2^(127-sb)
    uint32_t w0 = cvt_e4m3x2(v[0] * mul, v[1] * mul);
    uint32_t w1 = cvt_e4m3x2(v[2] * mul, v[3] * mul);
    uint32_t w2 = cvt_e4m3x2(v[4] * mul, v[5] * mul);
    uint32_t w3 = cvt_e4m3x2(v[6] * mul, v[7] * mul);
    q = make_uint2(w0 | (w1 << 16), w2 | (w3 << 16));
    scale = static_cast<uint32_t>(sb);
}

// Packs the scale bytes of the four blocks held by lanes 0,4,8,12 (and
// 16,20,24,28) into one little-endian word, valid in lanes 0 and 16.
__device__ __forceinline__ uint32_t gather_scale_word(uint32_t scale) {
    uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, scale, 4);
    uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, scale, 8);
    uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, scale, 12);
    return scale | (s1 << 8) | (s2 << 16) | (s3 << 24);
}

// One lane quantizes a whole 32-block held in 16 registers of packed BF16
// (same arithmetic as quantize_lane8, without shuffles).  Writes the 32 E4M3
// bytes into q[0..7] (little-endian words) and returns the scale byte.
__device__ __forceinline__ uint32_t quantize_block32(const uint4 (&raw)[4], uint32_t (&q)[8]) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        w[4 * i] = raw[i].x; w[4 * i + 1] = raw[i].y; w[4 * i + 2] = raw[i].z; w[4 * i + 3] = raw[i].w;
    }
    // amax magnitude as a BF16 bit pattern: per-halfword unsigned max of the
    // sign-cleared pairs, as a balanced tree.
    uint32_t m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = __vmaxu2(w[2 * i] & 0x7FFF7FFFu, w[2 * i + 1] & 0x7FFF7FFFu);
#pragma unroll
    for (int d = 1; d < 8; d <<= 1)
#pragma unroll
        for (int i = 0; i < 8; i += 2 * d) m[i] = __vmaxu2(m[i], m[i + d]);
    const uint32_t a = max(m[0] & 0xFFFFu, m[0] >> 16) << 16;  // FP32 bits of |amax|
    if (a >= 0x7F800000u) {  // Inf or NaN somewhere in the block
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = 0x7F7F7F7Fu;
        return 0xFFu;
    }
    int sb = static_cast<int>(a >> 23) - 8;
    sb = sb < 0 ? 0 : sb;
    const float mul = __uint_as_float(static_cast<uint32_t>(254 - sb) << 23);  // 2^(127-sb)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t lo = cvt_e4m3x2(__uint_as_float(w[2 * i] << 16) * mul,
                                       __uint_as_float(w[2 * i] & 0xFFFF0000u) * mul);
        const uint32_t hi = cvt_e4m3x2(__uint_as_float(w[2 * i + 1] << 16) * mul,
                                       __uint_as_float(w[2 * i + 1] & 0xFFFF0000u) * mul);
        q[i] = lo | (hi << 16);
    }
    return static_cast<uint32_t>(sb);
}

__device__ __forceinline__ void bf16x8_to_float(const uint4& raw, float (&v)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

}  // namespace mxk
