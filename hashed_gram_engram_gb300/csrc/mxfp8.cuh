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

}  // namespace engram
