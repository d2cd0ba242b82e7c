// Gate and masked residual: the arithmetic of _engram_gate_finish_kernel
// ("vllm.models.deepseek_v41.amd.engram") with one rank, which is the
// generic post-wkv kernel of Engram.forward
// ("vllm.models.deepseek_v4_1.common.engram"):
//   hr   = rsqrt(sum_d hidden^2 / D + eps)
//   kr   = rsqrt(sum_d key^2 / D + eps)
//   dot  = sum_d(hidden * q * k * key) * hr * kr / sqrt(D)
//   gate = sigmoid(sign(dot) * sqrt(max(|dot|, clamp)))      (0 if masked)
//   out  = hidden + gate * value          (masked tokens: hidden's bits)
// One CTA per token handles all hc copies, so the shared value is read
// once.  The per-token sums are reduced in a fixed order (shuffle tree,
// then warps in index order) and the run is deterministic.
//
// The key sums come as per-key-tile partials (sum key^2,
// sum hidden*q*k*key) written by the wkv epilogue, the value as bf16.
// Hidden is read before the programmatic-launch wait, so its HBM read
// overlaps the tail of the wkv kernel.
#include "internal.h"
#include "ptx.cuh"

namespace engram {
namespace {

constexpr int kMaxChunks = 2;    // 16-byte chunks of one row per thread
constexpr int kGateThreads = 512; // so D <= 8192

struct GateArgs {
    const uint16_t* hidden;
    int64_t hs_t, hs_h;
    uint16_t* out;
    int64_t os_t, os_h;
    const uint8_t* mask;
    const float* qk;  // [H, D]
    float* gate_out;  // [T, H]
    int T, D;
    float eps, clamp, inv_d, inv_sqrt_d;
    const float2* partials;
    const uint16_t* value;
    int J;
};

template <int H>
__global__ void __launch_bounds__(kGateThreads) gate_residual_kernel(const GateArgs a) {
    __shared__ float red[kGateThreads / 32][H];
    __shared__ float gate_s[H];
    const int t = blockIdx.x;
    const int tid = threadIdx.x;
    const int nchunk = a.D >> 3;
    const bool active = a.mask == nullptr || a.mask[t] != 0;

    float shh[H];
#pragma unroll
    for (int h = 0; h < H; ++h) shh[h] = 0.f;
    uint4 hid[kMaxChunks][H];
    float val[kMaxChunks][8];

    // Phase 1 (inputs only): hidden rows and sum hidden^2.
#pragma unroll
    for (int ci = 0; ci < kMaxChunks; ++ci) {
        const int c = tid + ci * blockDim.x;
        if (c < nchunk) {
#pragma unroll
            for (int h = 0; h < H; ++h) {
                hid[ci][h] = ld_nc_v4(a.hidden + t * a.hs_t + h * a.hs_h + c * 8);
                const uint32_t w[4] = {hid[ci][h].x, hid[ci][h].y, hid[ci][h].z, hid[ci][h].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float x0 = bf16lo(w[i]), x1 = bf16hi(w[i]);
                    shh[h] = fmaf(x0, x0, shh[h]);
                    shh[h] = fmaf(x1, x1, shh[h]);
                }
            }
        }
    }

    pdl_wait();  // the projection is complete and visible past this point

    // Phase 2: the value.
#pragma unroll
    for (int ci = 0; ci < kMaxChunks; ++ci) {
        const int c = tid + ci * blockDim.x;
        if (c < nchunk) {
            const int d = c * 8;
            const uint4 vb = ld_nc_v4(a.value + static_cast<int64_t>(t) * a.D + d);
            const uint32_t w[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
                val[ci][i] = (i & 1) ? bf16hi(w[i >> 1]) : bf16lo(w[i >> 1]);
        }
    }

    // Block reduction in a fixed order.
    const int lane = tid & 31, warp = tid >> 5, nwarps = (blockDim.x + 31) >> 5;
#pragma unroll
    for (int h = 0; h < H; ++h) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            shh[h] += __shfl_xor_sync(0xFFFFFFFFu, shh[h], off);
    }
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < H; ++h) red[warp][h] = shh[h];
    }
    __syncthreads();
    if (tid < H) {
        const int h = tid;
        float s_hh = 0.f, s_kk = 0.f, s_hk = 0.f;
        for (int w = 0; w < nwarps; ++w) s_hh += red[w][h];
        const float2* p = a.partials + (static_cast<int64_t>(t) * H + h) * a.J;
        for (int j = 0; j < a.J; ++j) {
            const float2 v = p[j];
            s_kk += v.x;
            s_hk += v.y;
        }
        const float hr = 1.0f / sqrtf(s_hh * a.inv_d + a.eps);
        const float kr = 1.0f / sqrtf(s_kk * a.inv_d + a.eps);
        const float dot = s_hk * hr * kr * a.inv_sqrt_d;
        float gi = sqrtf(fmaxf(fabsf(dot), a.clamp));
        if (dot < 0.0f) gi = -gi;
        float g = 1.0f / (1.0f + expf(-gi));
        if (!active) g = 0.0f;
        gate_s[h] = g;
        a.gate_out[static_cast<int64_t>(t) * H + h] = g;
    }
    __syncthreads();

    // Phase 3: the residual update.
#pragma unroll
    for (int ci = 0; ci < kMaxChunks; ++ci) {
        const int c = tid + ci * blockDim.x;
        if (c < nchunk) {
#pragma unroll
            for (int h = 0; h < H; ++h) {
                uint4 o = hid[ci][h];
                if (active) {
                    const float g = gate_s[h];
                    const uint32_t w[4] = {o.x, o.y, o.z, o.w};
                    uint32_t r[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        r[i] = pack_bf16x2(fmaf(g, val[ci][2 * i], bf16lo(w[i])),
                                           fmaf(g, val[ci][2 * i + 1], bf16hi(w[i])));
                    o = make_uint4(r[0], r[1], r[2], r[3]);
                }
                st_v4(a.out + t * a.os_t + h * a.os_h + c * 8, o);
            }
        }
    }
}

__global__ void qk_kernel(const uint16_t* q, const uint16_t* k, float* qk, int64_t n) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < n) qk[i] = __uint_as_float(static_cast<uint32_t>(q[i]) << 16) *
                       __uint_as_float(static_cast<uint32_t>(k[i]) << 16);
}

// fp32 value [T, D] of the last forward, for validation.
__global__ void debug_value_kernel(const uint16_t* value, int64_t n, float* out) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < n) out[i] = __uint_as_float(static_cast<uint32_t>(value[i]) << 16);
}

cudaError_t launch_gate(const engram_handle* h, const void* hidden, const int64_t* hs,
                        const uint8_t* mask, void* out, const int64_t* os, int64_t T,
                        cudaStream_t s, bool pdl) {
    GateArgs a = {};
    a.hidden = static_cast<const uint16_t*>(hidden);
    a.hs_t = hs[0];
    a.hs_h = hs[1];
    a.out = static_cast<uint16_t*>(out);
    a.os_t = os[0];
    a.os_h = os[1];
    a.mask = mask;
    a.qk = h->ws.qk;
    a.gate_out = h->ws.gate;
    a.T = static_cast<int>(T);
    a.D = static_cast<int>(h->cfg.dim);
    a.eps = static_cast<float>(h->cfg.eps);
    a.clamp = static_cast<float>(h->cfg.clamp);
    a.inv_d = 1.0f / static_cast<float>(a.D);
    a.inv_sqrt_d = 1.0f / sqrtf(static_cast<float>(a.D));
    a.partials = h->ws.partials;
    a.value = h->ws.value;
    a.J = a.D / prefill_bn(h);

    int threads = a.D / 8;
    if (threads > kGateThreads) threads = kGateThreads;
    threads = (threads + 31) / 32 * 32;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(T));
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    switch (h->cfg.hc_mult) {
        case 1: return cudaLaunchKernelEx(&cfg, gate_residual_kernel<1>, a);
        case 2: return cudaLaunchKernelEx(&cfg, gate_residual_kernel<2>, a);
        case 3: return cudaLaunchKernelEx(&cfg, gate_residual_kernel<3>, a);
        case 4: return cudaLaunchKernelEx(&cfg, gate_residual_kernel<4>, a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_gate_from_partials(const engram_handle* h, const void* hidden,
                                      const int64_t* hs, const uint8_t* mask, void* out,
                                      const int64_t* os, int64_t T, cudaStream_t s, bool pdl) {
    return launch_gate(h, hidden, hs, mask, out, os, T, s, pdl);
}

cudaError_t launch_qk(const engram_handle* h, cudaStream_t s) {
    const int64_t n = h->cfg.hc_mult * h->cfg.dim;
    qk_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(h->q, h->k, h->ws.qk, n);
    return cudaGetLastError();
}

cudaError_t launch_debug_value(const engram_handle* h, float* value, int64_t T, cudaStream_t s) {
    const int64_t n = T * h->cfg.dim;
    debug_value_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(h->ws.value, n,
                                                                              value);
    return cudaGetLastError();
}

}  // namespace engram
