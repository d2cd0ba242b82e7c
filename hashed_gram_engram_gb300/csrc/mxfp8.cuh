// MXFP8 activation quantisation shared by the gather kernels: per 32
// consecutive k, the E8M0 scale 2^e with e the smallest integer such that the
// block's largest magnitude is at most 448 * 2^e (e = 0 for an all-zero
// block, clamped to [-127, 127]), and e4m3 codes of x / 2^e rounded to
// nearest even with saturation (OCP MX v1.0 e4m3, E8M0).  x / 2^e is exact
// in fp32 for bf16 x, so the codes are the exact rounding of x / 2^e.
#pragma once

#include <cuda_fp8.h>

#include "ptx.cuh"

namespace engram {

// 448 = 1.75 * 2^8: for amax = 1.m * 2^u the answer is u - 8, plus one when
// 1.m > 1.75.
__device__ __forceinline__ int mx_scale_exponent(float amax) {
    const uint32_t b = __float_as_uint(amax);
    const int ef = static_cast<int>((b >> 23) & 0xFFu);
    if (ef == 0) return (b & 0x7FFFFFu) ? -127 : 0;
    int e = ef - 127 - 8 + (((b & 0x7FFFFFu) > 0x600000u) ? 1 : 0);
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// Four e4m3 codes of 4 bf16 (two packed words) times 2^-e.
__device__ __forceinline__ uint32_t mx_codes4(uint32_t w0, uint32_t w1, float inv) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(bf16lo(w0) * inv, bf16hi(w0) * inv), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(bf16lo(w1) * inv, bf16hi(w1) * inv), __NV_SATFINITE, __NV_E4M3);
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// 32 bf16 (four 16-byte chunks) -> 32 e4m3 codes (two 16-byte chunks);
// returns the biased E8M0 scale byte.
__device__ __forceinline__ uint32_t mx_quantize32(const uint4 (&v)[4], uint4 (&codes)[2]) {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            m = max(m, w[j] & 0x7FFFu);
            m = max(m, (w[j] >> 16) & 0x7FFFu);
        }
    }
    const int e = mx_scale_exponent(__uint_as_float(m << 16));
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint4 a = v[2 * h], b = v[2 * h + 1];
        codes[h] = make_uint4(mx_codes4(a.x, a.y, inv), mx_codes4(a.z, a.w, inv),
                              mx_codes4(b.x, b.y, inv), mx_codes4(b.z, b.w, inv));
    }
    return static_cast<uint32_t>(e + 127);
}

// ---------------------------------------------------------------- fp8 tables
// Rows of an fp8 table (class ParallelEngramEmbedding): e4m3 codes with one
// E8M0 scale byte per 32 elements, dequantized to bf16 on lookup:
// e4m3(code) * 2^(scale - 127), rounded to bf16 (nearest, ties to even).

// OCP e4m3 ("fn"): sign, 4-bit exponent with bias 7, 3-bit mantissa;
// exponent 0 holds the subnormals m * 2^-9; S.1111.111 is NaN (no inf).
__device__ __forceinline__ float e4m3_value(uint32_t b) {
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    float v;
    if (e == 0u)
        v = static_cast<float>(m) * 0x1p-9f;
    else if (e == 15u && m == 7u)
        v = __uint_as_float(0x7FC00000u);
    else
        v = __uint_as_float(((e + 120u) << 23) | (m << 20));  // (1 + m/8) * 2^(e-7)
    return (b & 0x80u) ? -v : v;
}

// E8M0 byte s -> 2^(s - 127) as fp32 (s = 0: the subnormal 2^-127; 255: NaN).
__device__ __forceinline__ float e8m0_value(uint32_t s) {
    if (s == 0u) return __uint_as_float(0x00400000u);
    if (s == 255u) return __uint_as_float(0x7FC00000u);
    return __uint_as_float(s << 23);
}

// Eight e4m3 codes (a 64-bit word, lowest byte first) times one block
// scale -> eight bf16 in a 16-byte chunk.  Each product is exact in fp32
// (four significant bits times a power of two), so the one rounding is the
// bf16 conversion.
__device__ __forceinline__ uint4 dequant8(uint2 codes, uint32_t scale_byte) {
    const float sc = e8m0_value(scale_byte);
    const uint32_t c[2] = {codes.x, codes.y};
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t q = c[i >> 1] >> (16 * (i & 1));
        w[i] = pack_bf16x2(e4m3_value(q & 0xFFu) * sc, e4m3_value((q >> 8) & 0xFFu) * sc);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace engram
