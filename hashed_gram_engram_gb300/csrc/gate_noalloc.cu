// engram_gate_noalloc: the gate and masked residual of Engram.forward
// ("vllm.models.deepseek_v4_1.common.engram") over a projection the caller
// computed, with no handle and no device allocation on any call.
//
// Who needs it: an inference engine that runs the wkv projection with its
// own GEMM (a library GEMM, or a column-sharded projection whose pieces it
// gathers itself) and only wants the gate stage.  Such engines size their
// KV-cache and activation pools to nearly all of HBM before serving and
// route every buffer through their own allocator; a library that calls
// cudaMalloc in the middle of a step can fail for lack of memory the engine
// has already claimed, and cudaMalloc/cudaFree synchronise the device,
// which stalls the engine's other streams.  So this entry point takes every
// buffer from the caller and keeps its one intermediate in a fixed device
// array that is part of the library image.
//
// The arithmetic is the split-dim form of the gate in
// "vllm.models.deepseek_v41.amd.engram" (_engram_gate_partials_kernel, then
// _engram_gate_finish_kernel), with the 256-dim slices of one device in
// place of tensor-parallel ranks:
//   partials: per (token, hc copy, 256-dim slice s) the three sums
//             (sum hidden^2, sum key^2, sum hidden*q*k*key) over the slice
//   finish:   per token, the slice sums are added in slice order, then
//             gate = sigmoid(sign(dot) * sqrt(max(|dot|, clamp))) with
//             dot = s_hk * rsqrt(s_hh/D + eps) * rsqrt(s_kk/D + eps) / sqrt(D),
//             and out = hidden + gate * value (masked tokens: hidden's bits).
//
// Scratch: g_partials below, kNoallocMaxPartials float4 slots (2 MiB), one
// per (token, hc copy, slice); a call needs T * H * (D / 256) of them and is
// refused with ENGRAM_ERR_SCRATCH_LIMIT beyond that.  No slot has to start at
// zero: the partials kernel of a call writes every slot that call's finish
// kernel reads, earlier on the same stream.  Because there is one array per
// device, two calls whose kernels can run at the same time on one device
// (two streams without an ordering between them, or two host threads)
// overwrite each other's partials; callers order their calls.  The array's
// device address is looked up once per device, on the first call there (a
// T = 0 call does only this), which may also load the library's device code
// onto that device: make that first call before capturing a stream.
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace engram {
namespace {

constexpr int kNoallocMaxPartials = 131072;  // 2 MiB of float4
constexpr int kSlice = 256;                  // dims per partial: 32 lanes x 8
constexpr int kPartialWarps = 4;             // (token, slice) pairs per CTA
constexpr int kFinishThreads = 512;          // so D <= 8192 with 2 chunks a thread
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float4 g_partials[kNoallocMaxPartials];

struct NoallocArgs {
    const uint16_t* hidden;
    int64_t hs_t, hs_h;
    const uint16_t* kv;
    int64_t kv_t;
    const uint16_t* q;
    const uint16_t* k;
    const uint8_t* mask;
    uint16_t* out;
    int64_t os_t, os_h;
    float4* partials;
    int T, D, S;
    float eps, clamp, inv_d, inv_sqrt_d;
};

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = bf16lo(w[i]);
        f[2 * i + 1] = bf16hi(w[i]);
    }
}

// One warp per (token, slice); lane l covers dims [256 s + 8 l, +8).
template <int H>
__global__ void __launch_bounds__(kPartialWarps * 32) noalloc_partials_kernel(const NoallocArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t pair = static_cast<int64_t>(blockIdx.x) * kPartialWarps + (threadIdx.x >> 5);
    if (pair >= static_cast<int64_t>(a.T) * a.S) return;
    const int t = static_cast<int>(pair / a.S);
    const int s = static_cast<int>(pair - static_cast<int64_t>(t) * a.S);
    const int d = s * kSlice + lane * 8;
#pragma unroll
    for (int h = 0; h < H; ++h) {
        float x[8], key[8], qv[8], kw[8];
        unpack8(ld_nc_v4(a.hidden + t * a.hs_t + h * a.hs_h + d), x);
        unpack8(ld_nc_v4(a.kv + t * a.kv_t + static_cast<int64_t>(h) * a.D + d), key);
        unpack8(ld_nc_v4(a.q + h * a.D + d), qv);
        unpack8(ld_nc_v4(a.k + h * a.D + d), kw);
        float shh = 0.f, skk = 0.f, shk = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            shh = fmaf(x[i], x[i], shh);
            skk = fmaf(key[i], key[i], skk);
            shk = fmaf(x[i] * (qv[i] * kw[i]), key[i], shk);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            shh += __shfl_xor_sync(0xFFFFFFFFu, shh, off);
            skk += __shfl_xor_sync(0xFFFFFFFFu, skk, off);
            shk += __shfl_xor_sync(0xFFFFFFFFu, shk, off);
        }
        if (lane == 0)
            a.partials[(static_cast<int64_t>(t) * H + h) * a.S + s] = make_float4(shh, skk, shk, 0.f);
    }
}

// One CTA per token: the gate of each hc copy, then the residual update.
template <int H>
__global__ void __launch_bounds__(kFinishThreads) noalloc_finish_kernel(const NoallocArgs a) {
    __shared__ float gate_s[H];
    const int t = blockIdx.x;
    const int tid = threadIdx.x;
    const bool active = a.mask == nullptr || a.mask[t] != 0;
    if (tid < H) {
        const float4* p = a.partials + (static_cast<int64_t>(t) * H + tid) * a.S;
        float s_hh = 0.f, s_kk = 0.f, s_hk = 0.f;
        for (int s = 0; s < a.S; ++s) {
            const float4 v = p[s];
            s_hh += v.x;
            s_kk += v.y;
            s_hk += v.z;
        }
        const float hr = 1.0f / sqrtf(s_hh * a.inv_d + a.eps);
        const float kr = 1.0f / sqrtf(s_kk * a.inv_d + a.eps);
        const float dot = s_hk * hr * kr * a.inv_sqrt_d;
        float gi = sqrtf(fmaxf(fabsf(dot), a.clamp));
        if (dot < 0.0f) gi = -gi;
        gate_s[tid] = active ? 1.0f / (1.0f + expf(-gi)) : 0.0f;
    }
    __syncthreads();
    const int nchunk = a.D >> 3;
    for (int c = tid; c < nchunk; c += blockDim.x) {
        float v[8];
        unpack8(ld_nc_v4(a.kv + t * a.kv_t + static_cast<int64_t>(H) * a.D + c * 8), v);
#pragma unroll
        for (int h = 0; h < H; ++h) {
            uint4 o = ld_nc_v4(a.hidden + t * a.hs_t + h * a.hs_h + c * 8);
            if (active) {
                const float g = gate_s[h];
                const uint32_t w[4] = {o.x, o.y, o.z, o.w};
                uint32_t r[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    r[i] = pack_bf16x2(fmaf(g, v[2 * i], bf16lo(w[i])),
                                       fmaf(g, v[2 * i + 1], bf16hi(w[i])));
                o = make_uint4(r[0], r[1], r[2], r[3]);
            }
            st_v4(a.out + t * a.os_t + h * a.os_h + c * 8, o);
        }
    }
}

template <int H>
cudaError_t launch_noalloc(const NoallocArgs& a, cudaStream_t s) {
    const int64_t pairs = static_cast<int64_t>(a.T) * a.S;
    noalloc_partials_kernel<H><<<static_cast<unsigned>((pairs + kPartialWarps - 1) / kPartialWarps),
                                 kPartialWarps * 32, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    int threads = a.D / 8;
    if (threads > kFinishThreads) threads = kFinishThreads;
    noalloc_finish_kernel<H><<<static_cast<unsigned>(a.T), threads, 0, s>>>(a);
    return cudaGetLastError();
}

// Device address of g_partials: looked up on the first call on a device and
// again whenever the context current on that device changes (after a
// cudaDeviceReset the primary context is a new one, and a caller may make a
// context of its own current), so a stale address is never passed to a
// kernel.  Contexts are told apart by their driver-assigned unique id; if
// the driver cannot report one, the address is looked up on every call.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <class Fn>
Fn driver_fn(const char* name) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<Fn>(p);
    return nullptr;
}

bool current_context_id(unsigned long long* id) {
    static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (get_current == nullptr || get_id == nullptr) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

struct ScratchEntry {
    unsigned long long ctx_id;
    void* addr;
};
std::mutex g_scratch_mu;
ScratchEntry g_scratch[kMaxDevices] = {};

cudaError_t scratch_address(int dev, void** out) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    unsigned long long id = 0;
    const bool known = current_context_id(&id);
    if (!known || g_scratch[dev].addr == nullptr || g_scratch[dev].ctx_id != id) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_partials);
        if (e != cudaSuccess) return e;
        // (the lookup initialises the device's primary context if it was not yet)
        if (current_context_id(&id)) {
            g_scratch[dev].ctx_id = id;
            g_scratch[dev].addr = p;
        } else {
            g_scratch[dev].addr = nullptr;  // no id to key on: look up every call
        }
        *out = p;
        return cudaSuccess;
    }
    *out = g_scratch[dev].addr;
    return cudaSuccess;
}

bool bad_view(const void* p, const int64_t* st) {
    return p == nullptr || st == nullptr || st[0] < 0 || st[1] < 0 || st[2] != 1 ||
           (reinterpret_cast<uintptr_t>(p) & 15u) != 0 || st[0] % 8 != 0 || st[1] % 8 != 0;
}

// A [T, H, D] view (unit dim stride) whose T*H rows of D elements are
// disjoint: rows nested copy-inside-token or token-inside-copy.  An output
// whose rows overlap would be written by several threads at once.
bool rows_disjoint(const int64_t* st, int64_t T, int64_t H, int64_t D) {
    if (H == 1) return T == 1 || st[0] >= D;
    if (T == 1) return st[1] >= D;
    return (st[1] >= D && st[0] >= H * st[1]) || (st[0] >= D && st[1] >= T * st[0]);
}

// Bytes spanned by a [T, H, D] bf16 view (non-negative strides, d stride 1).
int64_t span(const int64_t* st, int64_t T, int64_t H, int64_t D) {
    return ((T - 1) * st[0] + (H - 1) * st[1] + D) * 2;
}

bool overlap(const void* a, int64_t an, const void* b, int64_t bn) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + static_cast<uintptr_t>(bn) && pb < pa + static_cast<uintptr_t>(an);
}

}  // namespace
}  // namespace engram

extern "C" int engram_gate_noalloc(const void* hidden, const int64_t hidden_strides[3],
                                   const void* kv, int64_t kv_row_stride, const void* q_weight,
                                   const void* k_weight, const uint8_t* token_mask, void* out,
                                   const int64_t out_strides[3], int64_t T, int64_t H, int64_t D,
                                   double eps, double clamp, cudaStream_t stream) {
    using namespace engram;
    if (T < 0 || H < 1 || H > 4 || D < kSlice || D % kSlice != 0 || D > 8192 || !(eps >= 0.0) ||
        !(clamp >= 0.0))
        return ENGRAM_ERR_INVALID_ARG;
    if (T > 0) {
        if (bad_view(hidden, hidden_strides) || bad_view(out, out_strides) || kv == nullptr ||
            q_weight == nullptr || k_weight == nullptr || kv_row_stride < (H + 1) * D ||
            kv_row_stride % 8 != 0 || ((reinterpret_cast<uintptr_t>(kv) |
                                        reinterpret_cast<uintptr_t>(q_weight) |
                                        reinterpret_cast<uintptr_t>(k_weight)) & 15u) != 0)
            return ENGRAM_ERR_INVALID_ARG;
        // out's rows must not overlap each other; out may be hidden itself
        // (same strides) but overlap no other input
        const int64_t ob = span(out_strides, T, H, D);
        const bool in_place = out == hidden && out_strides[0] == hidden_strides[0] &&
                              out_strides[1] == hidden_strides[1];
        if (!rows_disjoint(out_strides, T, H, D) ||
            (!in_place && overlap(out, ob, hidden, span(hidden_strides, T, H, D))) ||
            overlap(out, ob, kv, ((T - 1) * kv_row_stride + (H + 1) * D) * 2) ||
            overlap(out, ob, q_weight, H * D * 2) || overlap(out, ob, k_weight, H * D * 2) ||
            (token_mask != nullptr && overlap(out, ob, token_mask, T)))
            return ENGRAM_ERR_INVALID_ARG;
        if (T > kNoallocMaxPartials || T * H * (D / kSlice) > kNoallocMaxPartials)
            return ENGRAM_ERR_SCRATCH_LIMIT;
    }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return ENGRAM_ERR_CUDA;
    void* scratch = nullptr;
    if (scratch_address(dev, &scratch) != cudaSuccess) return ENGRAM_ERR_CUDA;
    if (T == 0) return ENGRAM_OK;

    NoallocArgs a = {};
    a.hidden = static_cast<const uint16_t*>(hidden);
    a.hs_t = hidden_strides[0];
    a.hs_h = hidden_strides[1];
    a.kv = static_cast<const uint16_t*>(kv);
    a.kv_t = kv_row_stride;
    a.q = static_cast<const uint16_t*>(q_weight);
    a.k = static_cast<const uint16_t*>(k_weight);
    a.mask = token_mask;
    a.out = static_cast<uint16_t*>(out);
    a.os_t = out_strides[0];
    a.os_h = out_strides[1];
    a.partials = static_cast<float4*>(scratch);
    a.T = static_cast<int>(T);
    a.D = static_cast<int>(D);
    a.S = static_cast<int>(D / kSlice);
    a.eps = static_cast<float>(eps);
    a.clamp = static_cast<float>(clamp);
    a.inv_d = 1.0f / static_cast<float>(D);
    a.inv_sqrt_d = 1.0f / sqrtf(static_cast<float>(D));
    cudaError_t e;
    switch (H) {
        case 1: e = launch_noalloc<1>(a, stream); break;
        case 2: e = launch_noalloc<2>(a, stream); break;
        case 3: e = launch_noalloc<3>(a, stream); break;
        default: e = launch_noalloc<4>(a, stream); break;
    }
    return e == cudaSuccess ? ENGRAM_OK : ENGRAM_ERR_CUDA;
}
