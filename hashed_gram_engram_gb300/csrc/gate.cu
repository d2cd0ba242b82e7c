// Gate and masked residual: the arithmetic of _engram_gate_finish_kernel
// ("vllm.models.deepseek_v41.amd.engram") with one rank, which is the
// generic post-wkv kernel of Engram.forward
// ("vllm.models.deepseek_v4_1.common.engram"):
//   hr   = rsqrt(sum_d hidden^2 / D + eps)
//   kr   = rsqrt(sum_d key^2 / D + eps)
//   dot  = sum_d(hidden * q * k * key) * hr * kr / sqrt(D)
//   gate = sigmoid(sign(dot) * sqrt(max(|dot|, clamp)))      (0 if masked)
//   out  = hidden + gate * value          (masked tokens: hidden's bits)
//
// The three sums come as per-key-tile partials (sum hidden^2, sum key^2,
// sum hidden*q*k*key) written by the wkv epilogue, which reads hidden at
// the key columns anyway; the value comes as bf16.  What is left is a
// stream: per token, H hidden rows and the value row in, H rows out.
//
// gate_ring_kernel: persistent CTAs (two per SM when two token stages fit
// in half of the SM's shared memory, else one) take tokens c, c + grid, ...
// One thread (warp 8) keeps a ring of token stages full with bulk copies
// (the hidden rows, the value row, the token's partials) and writes each
// finished token back with bulk stores; warps 0-7 sum the partials of
// every copy in a fixed order (lane-strided, then a shuffle tree: runs are
// bit-identical), compute the gates and update the hidden rows in place in
// shared memory.  The hidden rows of the first stages are requested before
// the programmatic-launch wait, so their reads overlap the wkv kernel's tail.
//
// engram_forward accepts only 16-byte aligned rows, so every row is one
// bulk copy away; the largest configuration (D = 8192, H = 4) still gets two
// stages.
#include "internal.h"
#include "ptx.cuh"

namespace engram {
namespace {

constexpr int kRingCompute = 256;                 // warps 0-7
constexpr int kRingThreads = kRingCompute + 32;   // + warp 8: the copies
constexpr int kRingMaxStages = 8;
constexpr uint32_t kRingSmem = 227 * 1024;        // dynamic shared memory: one CTA per SM
constexpr uint32_t kRingSmemHalf = 113 * 1024;    // ... or two, when two stages fit in half
constexpr uint32_t kRingTail = 512;               // barriers, gates, flag, alignment

struct RingArgs {
    const uint16_t* hidden;
    int64_t hs_t, hs_h;
    uint16_t* out;
    int64_t os_t, os_h;
    const uint8_t* mask;
    const uint16_t* value;    // [T, D] bf16
    const float4* partials;   // [T, H, J]
    float* gate_out;          // [T, H]
    int T, D, H, J, stages;
    uint32_t row_bytes;       // D * 2
    uint32_t val_off, part_off, stage_bytes;
    float eps, clamp, inv_d, inv_sqrt_d;
    unsigned* err;
};

__device__ __forceinline__ float gate_of(float s_hh, float s_kk, float s_hk, float inv_d,
                                         float eps, float inv_sqrt_d, float clamp) {
    const float hr = 1.0f / sqrtf(s_hh * inv_d + eps);
    const float kr = 1.0f / sqrtf(s_kk * inv_d + eps);
    const float dot = s_hk * hr * kr * inv_sqrt_d;
    float gi = sqrtf(fmaxf(fabsf(dot), clamp));
    if (dot < 0.0f) gi = -gi;
    return 1.0f / (1.0f + expf(-gi));
}

// x + g * v for eight bf16 pairs, rounded to bf16
__device__ __forceinline__ uint4 residual8(uint4 x, uint4 v, float g) {
    const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
    const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
    uint32_t r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        r[i] = pack_bf16x2(fmaf(g, bf16lo(vw[i]), bf16lo(xw[i])),
                           fmaf(g, bf16hi(vw[i]), bf16hi(xw[i])));
    return make_uint4(r[0], r[1], r[2], r[3]);
}

__global__ void __launch_bounds__(kRingThreads, 2) gate_ring_kernel(const RingArgs a) {
    extern __shared__ uint8_t ring_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(ring_raw) + 127) & ~static_cast<uintptr_t>(127));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.stages * a.stage_bytes);
    uint64_t* done = full + kRingMaxStages;
    float* g_s = reinterpret_cast<float*>(done + kRingMaxStages);  // this token's gates
    int* abort_flag = reinterpret_cast<int*>(g_s + kMaxCopies);
    const volatile int* abort_v = abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x;
    const int n = (a.T - static_cast<int>(blockIdx.x) + G - 1) / G;  // tokens of this CTA
    auto token = [&](int i) { return static_cast<int>(blockIdx.x) + i * G; };
    auto fail = [&]() {
        *reinterpret_cast<volatile int*>(abort_flag) = 1;
        atomicOr(a.err, ENGRAM_DEVERR_TIMEOUT);
    };

    if (tid == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&done[s], 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    int issued = 0;  // token stages requested (warp 8, lane 0)
    if (warp == kRingCompute / 32) {
        if (lane == 0) {
            const uint32_t in_bytes =
                static_cast<uint32_t>(a.H + 1) * a.row_bytes + static_cast<uint32_t>(a.H * a.J) * 16u;
            auto load_hidden = [&](int i) {
                const int s = i % a.stages, t = token(i);
                uint8_t* st = smem + s * a.stage_bytes;
                mbar_arrive_expect_tx(&full[s], in_bytes);
                if (a.hs_h == a.D)  // the token's rows are one block
                    bulk_load(st, a.hidden + t * a.hs_t, a.H * a.row_bytes, &full[s]);
                else
                    for (int h = 0; h < a.H; ++h)
                        bulk_load(st + h * a.row_bytes, a.hidden + t * a.hs_t + h * a.hs_h,
                                  a.row_bytes, &full[s]);
            };
            auto load_rest = [&](int i) {  // written by the wkv kernel
                const int s = i % a.stages, t = token(i);
                uint8_t* st = smem + s * a.stage_bytes;
                bulk_load(st + a.val_off, a.value + static_cast<int64_t>(t) * a.D, a.row_bytes,
                          &full[s]);
                bulk_load(st + a.part_off, a.partials + static_cast<int64_t>(t) * a.H * a.J,
                          static_cast<uint32_t>(a.H * a.J) * 16u, &full[s]);
            };
            const int first = n < a.stages ? n : a.stages;
            for (int i = 0; i < first; ++i) load_hidden(i);
            pdl_wait();
            for (int i = 0; i < first; ++i) load_rest(i);
            issued = first;
            bool ok = true;
            for (int j = 0; j < n; ++j) {
                const int s = j % a.stages, t = token(j);
                if (!mbar_wait_sleep(&done[s], static_cast<uint32_t>((j / a.stages) & 1), abort_v,
                                     32)) {
                    ok = false;
                    break;
                }
                const uint8_t* st = smem + s * a.stage_bytes;
                if (a.os_h == a.D)
                    bulk_store(a.out + t * a.os_t, st, a.H * a.row_bytes);
                else
                    for (int h = 0; h < a.H; ++h)
                        bulk_store(a.out + t * a.os_t + h * a.os_h, st + h * a.row_bytes,
                                   a.row_bytes);
                bulk_commit();
                // the stage takes token j + stages once the store has read it
                // (the compute warps go on with the tokens already in place)
                if (a.stages >= 4) {
                    const int next = j - 1 + a.stages;
                    if (j >= 1 && next < n) {
                        bulk_wait_read<1>();
                        load_hidden(next);
                        load_rest(next);
                        ++issued;
                    }
                } else if (j + a.stages < n) {
                    bulk_wait_read<0>();
                    load_hidden(j + a.stages);
                    load_rest(j + a.stages);
                    ++issued;
                }
            }
            bulk_wait<0>();  // every store has landed
            if (!ok) fail();
        }
    } else {
        const int nchunk = a.D >> 3;  // 16-byte chunks of a row
        for (int j = 0; j < n; ++j) {
            const int s = j % a.stages, t = token(j);
            uint8_t* st = smem + s * a.stage_bytes;
            const bool got = mbar_wait(&full[s], static_cast<uint32_t>((j / a.stages) & 1), abort_v);
            if (named_barrier_or(1, kRingCompute, !got || *abort_v)) {
                if (!got) fail();
                break;
            }
            const bool active = a.mask == nullptr || a.mask[t] != 0;
            if (warp < a.H) {
                const float4* p = reinterpret_cast<const float4*>(st + a.part_off) + warp * a.J;
                float s_hh = 0.f, s_kk = 0.f, s_hk = 0.f;
                for (int jj = lane; jj < a.J; jj += 32) {
                    const float4 v = p[jj];
                    s_hh += v.x;
                    s_kk += v.y;
                    s_hk += v.z;
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    s_hh += __shfl_xor_sync(0xFFFFFFFFu, s_hh, o);
                    s_kk += __shfl_xor_sync(0xFFFFFFFFu, s_kk, o);
                    s_hk += __shfl_xor_sync(0xFFFFFFFFu, s_hk, o);
                }
                if (lane == 0) {
                    const float g = active ? gate_of(s_hh, s_kk, s_hk, a.inv_d, a.eps,
                                                     a.inv_sqrt_d, a.clamp)
                                           : 0.0f;
                    g_s[warp] = g;
                    a.gate_out[static_cast<int64_t>(t) * a.H + warp] = g;
                }
            }
            named_barrier_sync(1, kRingCompute);
            if (active) {  // (masked tokens leave with hidden's bits)
                const uint4* vrow = reinterpret_cast<const uint4*>(st + a.val_off);
                for (int k = tid; k < a.H * nchunk; k += kRingCompute) {
                    const int h = k / nchunk, c = k - h * nchunk;
                    uint4* hp = reinterpret_cast<uint4*>(st + h * a.row_bytes) + c;
                    *hp = residual8(*hp, vrow[c], g_s[h]);
                }
            }
            fence_proxy_async_smem();  // the bulk stores read these rows
            named_barrier_sync(1, kRingCompute);
            if (tid == 0) mbar_arrive(&done[s]);
        }
    }
    __syncthreads();
    if (*abort_v && tid == kRingCompute) {
        // copies still in flight land before the shared memory goes
        for (int i = issued > a.stages ? issued - a.stages : 0; i < issued; ++i)
            mbar_wait(&full[i % a.stages], static_cast<uint32_t>((i / a.stages) & 1), nullptr);
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

// Stage layout of the ring: H hidden rows | value row | H * J partials.
uint32_t ring_stage_bytes(int64_t D, int64_t H, int64_t J) {
    return static_cast<uint32_t>((H + 1) * D * 2 + H * J * 16);
}

}  // namespace

cudaError_t gate_setup_attributes() {
    return cudaFuncSetAttribute(gate_ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kRingSmem));
}

cudaError_t launch_gate_from_partials(const engram_handle* h, const void* hidden,
                                      const int64_t* hs, const uint8_t* mask, void* out,
                                      const int64_t* os, int64_t T, cudaStream_t s, bool pdl) {
    const int D = static_cast<int>(h->cfg.dim), H = static_cast<int>(h->cfg.hc_mult);
    // wkv partial records per (token, copy): one per tile, MXFP8 one per half tile
    const int J = (h->cfg.wkv_format == ENGRAM_WKV_MXFP8 ? 2 : 1) * (D / prefill_bn(h));
    const float inv_d = 1.0f / static_cast<float>(D);
    const float inv_sqrt_d = 1.0f / sqrtf(static_cast<float>(D));
    const float eps = static_cast<float>(h->cfg.eps), clamp = static_cast<float>(h->cfg.clamp);
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;

    const uint32_t stage = ring_stage_bytes(D, H, J);
    // two CTAs per SM (two independent copy streams) when each still gets two
    // stages; one CTA with the whole shared memory otherwise
    const bool two = 2u * stage <= kRingSmemHalf - kRingTail;
    const uint32_t smem = two ? kRingSmemHalf : kRingSmem;
    const int stages_fit = static_cast<int>((smem - kRingTail) / stage);
    if (stages_fit < 2) return cudaErrorInvalidConfiguration;
    RingArgs a = {};
    a.hidden = static_cast<const uint16_t*>(hidden);
    a.hs_t = hs[0];
    a.hs_h = hs[1];
    a.out = static_cast<uint16_t*>(out);
    a.os_t = os[0];
    a.os_h = os[1];
    a.mask = mask;
    a.value = h->ws.value;
    a.partials = h->ws.partials;
    a.gate_out = h->ws.gate;
    a.T = static_cast<int>(T);
    a.D = D;
    a.H = H;
    a.J = J;
    a.stages = stages_fit < kRingMaxStages ? stages_fit : kRingMaxStages;
    a.row_bytes = static_cast<uint32_t>(D) * 2u;
    a.val_off = static_cast<uint32_t>(H) * a.row_bytes;
    a.part_off = a.val_off + a.row_bytes;
    a.stage_bytes = stage;
    a.eps = eps;
    a.clamp = clamp;
    a.inv_d = inv_d;
    a.inv_sqrt_d = inv_sqrt_d;
    a.err = h->ws.err;
    const int64_t ctas = static_cast<int64_t>(h->num_sms) * (two ? 2 : 1);
    const int64_t grid = T < ctas ? T : ctas;
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kRingThreads);
    cfg.dynamicSmemBytes = smem;
    return cudaLaunchKernelEx(&cfg, gate_ring_kernel, a);
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
