// Lookups of a decode step's Engram layers run ahead on a side stream.
//
// The prefetch page ("vllm.models.deepseek_v41.nvidia.specialized_decode.
// engram.prefetch", class EngramPrefetch with start / forward / join) and
// Engram.prepare_embeddings ("vllm.models.deepseek_v4_1.common.engram") stage
// every layer's hash rows as soon as the step's hash ids exist, so that a
// layer's forward waits only for its own rows.  With a host-offloaded table
// the rows cross the host link, and that latency leaves each layer's
// critical path.
//
// Host code only: the work is engram_lookup (background grid) on a stream
// this object owns, one event per layer, and engram_forward (hash_ids = NULL)
// on the caller's stream after a wait on that event.  No kernel of its own.
// Everything it records and waits on is stream-ordered, so a CUDA graph
// capture of start / forward / join on the caller's stream records the fork
// to the side stream and the joins back.
#include <cstring>
#include <new>

#include "internal.h"

using namespace engram;

struct engram_prefetch {
    int device;
    int32_t n;
    engram_t** layers;      // borrowed
    bool* pending;          // rows staged by the last start, not yet consumed
    cudaEvent_t* done;      // per layer: its lookup finished on the side stream
    cudaEvent_t start_ev;   // the caller's stream at start
    cudaStream_t side;
    int64_t T;              // tokens of the last start
    int32_t flags;
    uint16_t** kv;          // ENGRAM_PREFETCH_WKV: per layer bf16 [kv_rows, N]
    int64_t* kv_rows;
    bool* kv_ready;         // the last start ran this layer's wkv (else its lookup only)
};

namespace {

struct Guard {
    int prev = -1;
    bool ok = false;
    explicit Guard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        ok = (prev == dev) || cudaSetDevice(dev) == cudaSuccess;
    }
    ~Guard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

void release(engram_prefetch* p) {
    if (p == nullptr) return;
    if (p->done != nullptr)
        for (int32_t i = 0; i < p->n; ++i)
            if (p->done[i] != nullptr) cudaEventDestroy(p->done[i]);
    if (p->start_ev != nullptr) cudaEventDestroy(p->start_ev);
    if (p->side != nullptr) cudaStreamDestroy(p->side);
    if (p->kv != nullptr)
        for (int32_t i = 0; i < p->n; ++i)
            if (p->kv[i] != nullptr) cudaFree(p->kv[i]);
    delete[] p->kv;
    delete[] p->kv_rows;
    delete[] p->kv_ready;
    delete[] p->done;
    delete[] p->pending;
    delete[] p->layers;
    delete p;
}

}  // namespace

extern "C" {

int engram_prefetch_create(engram_t* const* layers, int32_t n_layers, int32_t flags,
                           engram_prefetch_t** out) {
    if (out == nullptr) return ENGRAM_ERR_INVALID_ARG;
    *out = nullptr;
    if (layers == nullptr || n_layers < 1 || (flags & ~ENGRAM_PREFETCH_WKV) != 0)
        return ENGRAM_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n_layers; ++i)
        if (layers[i] == nullptr) return ENGRAM_ERR_INVALID_ARG;
    const int dev = layers[0]->cfg.device;
    for (int32_t i = 1; i < n_layers; ++i)
        if (layers[i]->cfg.device != dev) return ENGRAM_ERR_INVALID_ARG;
    engram_prefetch* p = new (std::nothrow) engram_prefetch();
    if (p == nullptr) return ENGRAM_ERR_OOM;
    std::memset(static_cast<void*>(p), 0, sizeof(*p));
    p->device = dev;
    p->n = n_layers;
    p->T = -1;
    p->layers = new (std::nothrow) engram_t*[n_layers];
    p->pending = new (std::nothrow) bool[n_layers];
    p->done = new (std::nothrow) cudaEvent_t[n_layers];
    p->flags = flags;
    p->kv = new (std::nothrow) uint16_t*[n_layers];
    p->kv_rows = new (std::nothrow) int64_t[n_layers];
    p->kv_ready = new (std::nothrow) bool[n_layers];
    if (p->layers == nullptr || p->pending == nullptr || p->done == nullptr ||
        p->kv == nullptr || p->kv_rows == nullptr || p->kv_ready == nullptr) {
        release(p);
        return ENGRAM_ERR_OOM;
    }
    for (int32_t i = 0; i < n_layers; ++i) {
        p->layers[i] = layers[i];
        p->pending[i] = false;
        p->done[i] = nullptr;
        p->kv[i] = nullptr;
        p->kv_rows[i] = 0;
        p->kv_ready[i] = false;
    }
    Guard g(dev);
    cudaError_t e = g.ok ? cudaSuccess : cudaErrorInvalidDevice;
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->start_ev, cudaEventDisableTiming);
    for (int32_t i = 0; i < n_layers && e == cudaSuccess; ++i)
        e = cudaEventCreateWithFlags(&p->done[i], cudaEventDisableTiming);
    // wkv mode: a kv buffer per layer for the largest T its fused launch serves
    for (int32_t i = 0; i < n_layers && e == cudaSuccess && (flags & ENGRAM_PREFETCH_WKV); ++i) {
        const engram_handle* h = layers[i];
        const int64_t tmax = h->cfg.wkv_format == ENGRAM_WKV_MXFP8 ? kMaxFusedTMx : kMaxFusedT;
        p->kv_rows[i] = h->cfg.max_tokens < tmax ? h->cfg.max_tokens : tmax;
        if (h->fused.ok)
            e = cudaMalloc(reinterpret_cast<void**>(&p->kv[i]),
                           static_cast<size_t>(p->kv_rows[i] * h->N * 2));
    }
    if (e != cudaSuccess) {
        release(p);
        return e == cudaErrorMemoryAllocation ? ENGRAM_ERR_OOM : ENGRAM_ERR_CUDA;
    }
    *out = p;
    return ENGRAM_OK;
}

int engram_prefetch_destroy(engram_prefetch_t* p) {
    if (p == nullptr) return ENGRAM_OK;
    Guard g(p->device);
    if (p->side != nullptr) cudaStreamSynchronize(p->side);
    release(p);
    return ENGRAM_OK;
}

int engram_prefetch_start(engram_prefetch_t* p, const int32_t* const* hash_ids,
                          const int64_t* ids_row_stride, int64_t T, int background,
                          cudaStream_t stream) {
    if (p == nullptr || hash_ids == nullptr || ids_row_stride == nullptr || T < 0)
        return ENGRAM_ERR_INVALID_ARG;
    for (int32_t i = 0; i < p->n; ++i) {
        if (T > p->layers[i]->cfg.max_tokens) return ENGRAM_ERR_T_EXCEEDS_MAX;
        if (T > 0 && (hash_ids[i] == nullptr || ids_row_stride[i] < p->layers[i]->C))
            return ENGRAM_ERR_INVALID_ARG;
    }
    Guard g(p->device);
    if (!g.ok) return ENGRAM_ERR_CUDA;
    for (int32_t i = 0; i < p->n; ++i) p->pending[i] = false;
    p->T = T;
    // the side stream starts after everything already issued on the
    // caller's stream: the hash ids, and the previous step's forwards that
    // read the staged rows about to be overwritten
    cudaError_t e = cudaEventRecord(p->start_ev, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->side, p->start_ev, 0);
    if (e != cudaSuccess) return ENGRAM_ERR_CUDA;
    for (int32_t i = 0; i < p->n; ++i) {
        engram_handle* h = p->layers[i];
        // wkv mode, where the layer's fused launch serves T: gather and
        // projection here, only the gate and residual left for forward
        p->kv_ready[i] = p->kv[i] != nullptr && T > 0 && T <= p->kv_rows[i] &&
                         fused_supported(h, T);
        const int rc = p->kv_ready[i]
                           ? engram_wkv(h, hash_ids[i], ids_row_stride[i], p->kv[i], h->N, T,
                                        p->side)
                           : engram_lookup(h, hash_ids[i], ids_row_stride[i], T, background,
                                           p->side);
        if (rc != ENGRAM_OK) return rc;
        if (cudaEventRecord(p->done[i], p->side) != cudaSuccess) return ENGRAM_ERR_CUDA;
        p->pending[i] = true;
    }
    return ENGRAM_OK;
}

int engram_prefetch_forward(engram_prefetch_t* p, int32_t layer, const void* hidden,
                            const int64_t hidden_strides[3], const int32_t* hash_ids,
                            int64_t ids_row_stride, const uint8_t* token_mask, void* out,
                            const int64_t out_strides[3], int64_t T, cudaStream_t stream) {
    if (p == nullptr || layer < 0 || layer >= p->n) return ENGRAM_ERR_INVALID_ARG;
    engram_t* h = p->layers[layer];
    if (!p->pending[layer]) {
        // nothing staged ahead for this layer: the plain forward
        if (hash_ids == nullptr && T > 0) return ENGRAM_ERR_INVALID_ARG;
        return engram_forward(h, hidden, hidden_strides, hash_ids, ids_row_stride, token_mask,
                              out, out_strides, T, stream);
    }
    if (T != p->T) return ENGRAM_ERR_INVALID_ARG;
    Guard g(p->device);
    if (!g.ok) return ENGRAM_ERR_CUDA;
    if (cudaStreamWaitEvent(stream, p->done[layer], 0) != cudaSuccess) return ENGRAM_ERR_CUDA;
    p->pending[layer] = false;
    if (p->kv_ready[layer])  // the post-wkv kernel of EngramPrefetch.forward
        return engram_gate_noalloc(hidden, hidden_strides, p->kv[layer], h->N, h->q, h->k,
                                   token_mask, out, out_strides, T, h->cfg.hc_mult, h->cfg.dim,
                                   h->cfg.eps, h->cfg.clamp, stream);
    return engram_forward(h, hidden, hidden_strides, nullptr, 0, token_mask, out, out_strides, T,
                          stream);
}

int engram_prefetch_join(engram_prefetch_t* p, cudaStream_t stream) {
    if (p == nullptr) return ENGRAM_ERR_INVALID_ARG;
    Guard g(p->device);
    if (!g.ok) return ENGRAM_ERR_CUDA;
    for (int32_t i = 0; i < p->n; ++i) {
        if (!p->pending[i]) continue;
        if (cudaStreamWaitEvent(stream, p->done[i], 0) != cudaSuccess) return ENGRAM_ERR_CUDA;
        p->pending[i] = false;
    }
    return ENGRAM_OK;
}

int engram_prefetch_pending(const engram_prefetch_t* p, int32_t layer) {
    if (p == nullptr || layer < 0 || layer >= p->n) return ENGRAM_ERR_INVALID_ARG;
    return p->pending[layer] ? 1 : 0;
}

}  // extern "C"
