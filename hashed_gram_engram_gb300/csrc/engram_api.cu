// C ABI of the Engram forward: handle life cycle, argument checks, the
// workspace, TMA descriptors and the launch sequence of one call.
//
// The sequence of engram_forward (Engram.forward, with the gather of
// Engram.prepare_embeddings folded in when hash ids are given):
//   decode (T <= 256 and a column slice of <= 256 per CTA): one cooperative
//     kernel does gather, projection, gate and residual (decode_fused.cu);
//   prefill: gather (plain launch: ordered after everything before it on
//     the stream), wkv (programmatic dependent launch: weight tiles stream in
//     while the gather runs; token tiles wait for it), gate (programmatic
//     dependent launch: hidden is read while the wkv kernel drains).
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "internal.h"

using namespace engram;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    // initialised once, also when handles are created from several threads
    static const EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

// 2-D K-major operand [rows, cols] of `elem` bytes, box = 128 bytes of K x
// box_rows, 128-byte swizzle (the layout the tcgen05 descriptors expect).
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem, int64_t cols,
              int64_t rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * elem)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kKBlockBytes / elem),
                         static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rows of 512 bytes (MXFP8 scale atoms, as 128 x 4-byte words), box =
// box_rows whole rows, no swizzle: a TMA copy of atoms in their stored order.
bool make_atom_map(CUtensorMap* m, const void* base, int64_t rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {512};
    cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Keeps the caller's current device across an entry point.
struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        ok = (prev == dev) || cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <class T>
cudaError_t dalloc(T** p, size_t bytes, bool zero) {
    *p = nullptr;
    if (bytes == 0) return cudaSuccess;
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(p), bytes);
    if (e != cudaSuccess) {
        *p = nullptr;
        return e;
    }
    if (zero) e = cudaMemset(*p, 0, bytes);
    return e;
}

void free_handle(engram_handle* h) {
    if (h == nullptr) return;
    void* ptrs[] = {h->d_row_offset, h->d_rows,      h->ws.staged,   h->ws.staged_q,
                    h->ws.staged_s,  h->ws.partials, h->ws.value,
                    h->ws.gate,      h->ws.qk,       h->ws.wsf_atoms, h->ws.err,
                    h->ws.wpack,     h->ws.fpart,    h->ws.fvalue,   h->ws.grid_bar,
                    h->ws.host_hidden, h->ws.host_ids, h->ws.host_mask,
                    h->ws.pipe_hidden[0], h->ws.pipe_hidden[1], h->ws.pipe_ids[0],
                    h->ws.pipe_ids[1], h->ws.pipe_mask[0], h->ws.pipe_mask[1]};
    for (void* p : ptrs)
        if (p) cudaFree(p);
    for (int b = 0; b < 2; ++b)
        for (cudaEvent_t ev : {h->pipe_ev_in[b], h->pipe_ev_fwd[b], h->pipe_ev_out[b]})
            if (ev) cudaEventDestroy(ev);
    if (h->pipe_in) cudaStreamDestroy(h->pipe_in);
    if (h->pipe_out) cudaStreamDestroy(h->pipe_out);
    for (cudaEvent_t ev : h->ev)
        if (ev) cudaEventDestroy(ev);
    delete h;
}

int set_err(engram_handle* h, int code) {
    if (h) h->last_error = code;
    return code;
}

int cuda_err(engram_handle* h, cudaError_t e) {
    if (e == cudaSuccess) return set_err(h, ENGRAM_OK);
    return set_err(h, e == cudaErrorMemoryAllocation ? ENGRAM_ERR_OOM : ENGRAM_ERR_CUDA);
}

bool ranges_overlap(const void* a, int64_t a_bytes, const void* b, int64_t b_bytes) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + static_cast<uintptr_t>(b_bytes) && pb < pa + static_cast<uintptr_t>(a_bytes);
}

// Bytes spanned by a [T, H, D] bf16 view with non-negative strides.
int64_t span_bytes(const int64_t* s, int64_t T, int64_t H, int64_t D) {
    return ((T - 1) * s[0] + (H - 1) * s[1] + (D - 1) * s[2] + 1) * 2;
}

int check_view(const void* p, const int64_t* s) {
    if (p == nullptr || s == nullptr) return ENGRAM_ERR_INVALID_ARG;
    if (s[0] < 0 || s[1] < 0 || s[2] != 1) return s[2] != 1 && s[2] > 0 ? ENGRAM_ERR_UNSUPPORTED
                                                                        : ENGRAM_ERR_INVALID_ARG;
    if (!aligned16(p) || (s[0] % 8) != 0 || (s[1] % 8) != 0) return ENGRAM_ERR_UNSUPPORTED;
    return ENGRAM_OK;
}

// An output view's T*H rows of D elements must be disjoint (nested
// copy-inside-token or token-inside-copy): rows that overlap would be
// written by several threads at once.
bool rows_disjoint(const int64_t* s, int64_t T, int64_t H, int64_t D) {
    if (H == 1) return T == 1 || s[0] >= D;
    if (T == 1) return s[1] >= D;
    return (s[1] >= D && s[0] >= H * s[1]) || (s[0] >= D && s[1] >= T * s[0]);
}

}  // namespace

extern "C" {

int engram_layout(int64_t vocab_size, int32_t max_ngram_size, int32_t n_heads, int32_t n_layers,
                  int64_t* primes, int64_t* offsets) {
    if (vocab_size < 1 || max_ngram_size < 2 || n_heads < 1 || n_layers < 1 || !primes ||
        !offsets)
        return ENGRAM_ERR_INVALID_ARG;
    const int64_t cols = static_cast<int64_t>(max_ngram_size - 1) * n_heads;
    const int64_t total = cols * n_layers;
    auto is_prime = [](int64_t n) {
        if (n < 2) return false;
        if (n % 2 == 0) return n == 2;
        for (int64_t d = 3; d * d <= n; d += 2)
            if (n % d == 0) return false;
        return true;
    };
    int64_t used = 0;  // primes[0..used) are taken
    for (int32_t l = 0; l < n_layers; ++l) {
        for (int32_t o = 0; o < max_ngram_size - 1; ++o) {
            int64_t cur = vocab_size - 1;
            for (int32_t hd = 0; hd < n_heads; ++hd) {
                bool taken = true;
                while (taken) {
                    do ++cur; while (!is_prime(cur));
                    taken = false;
                    for (int64_t i = 0; i < used && !taken; ++i) taken = primes[i] == cur;
                }
                primes[used++] = cur;
            }
        }
        int64_t acc = 0;
        for (int64_t c = 0; c < cols; ++c) {
            offsets[l * cols + c] = acc;
            acc += primes[l * cols + c];
        }
    }
    (void)total;
    return ENGRAM_OK;
}

int engram_create(const engram_config* cfg, const engram_weights* w, engram_t** out) {
    if (out == nullptr) return ENGRAM_ERR_INVALID_ARG;
    *out = nullptr;
    if (cfg == nullptr || w == nullptr) return ENGRAM_ERR_INVALID_ARG;
    const engram_config c = *cfg;
    if (c.dim <= 0 || c.hc_mult <= 0 || c.max_ngram_size < 2 || c.n_heads < 1 ||
        c.head_dim <= 0 || c.max_tokens <= 0 || !(c.eps >= 0.0) || !(c.clamp >= 0.0) ||
        (c.table_format != ENGRAM_TABLE_FORMAT_BF16 && c.table_format != ENGRAM_TABLE_FORMAT_E4M3) ||
        (c.wkv_format != ENGRAM_WKV_BF16 && c.wkv_format != ENGRAM_WKV_MXFP8) ||
        (c.table_location != ENGRAM_TABLE_DEVICE && c.table_location != ENGRAM_TABLE_HOST_PINNED))
        return ENGRAM_ERR_INVALID_ARG;
    if (w->table == nullptr || w->row_offset == nullptr || w->rows == nullptr ||
        w->wkv == nullptr || w->q_weight == nullptr || w->k_weight == nullptr)
        return ENGRAM_ERR_INVALID_ARG;
    if (c.wkv_format == ENGRAM_WKV_MXFP8 && w->wkv_scale == nullptr) return ENGRAM_ERR_INVALID_ARG;
    const bool tfp8 = c.table_format == ENGRAM_TABLE_FORMAT_E4M3;
    if (tfp8 && w->table_scale == nullptr) return ENGRAM_ERR_INVALID_ARG;
    const int64_t C = (c.max_ngram_size - 1) * c.n_heads;
    const int64_t K = C * c.head_dim;
    const int64_t N = c.dim * (c.hc_mult + 1);
    // What the kernels are built for.
    const bool mx = c.wkv_format == ENGRAM_WKV_MXFP8;
    if (c.dim % kBNPrefill != 0 || c.dim > 8192 || c.hc_mult > 4 || c.head_dim % 8 != 0 ||
        32 % (c.head_dim / 8) != 0 || K % 128 != 0 || K > (1 << 20) || !aligned16(w->table) ||
        !aligned16(w->wkv) || c.max_tokens > (1 << 24) ||
        (mx && (c.head_dim % 32 != 0 || !aligned16(w->wkv_scale))) ||
        (tfp8 && c.head_dim % 32 != 0))
        return ENGRAM_ERR_UNSUPPORTED;
    for (int64_t i = 0; i < C; ++i)
        if (w->rows[i] <= 0 || w->row_offset[i] < 0) return ENGRAM_ERR_INVALID_ARG;

    DeviceGuard guard(c.device);
    if (!guard.ok) return ENGRAM_ERR_CUDA;
    int sms = 0, uva = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, c.device) != cudaSuccess ||
        cudaDeviceGetAttribute(&uva, cudaDevAttrUnifiedAddressing, c.device) != cudaSuccess)
        return ENGRAM_ERR_CUDA;

    const void* table = w->table;
    const void* table_scale = tfp8 ? static_cast<const void*>(w->table_scale) : nullptr;
    if (c.table_location == ENGRAM_TABLE_HOST_PINNED) {
        if (!uva) return ENGRAM_ERR_NO_UVA;
        // the device aliases of the pinned table (and of its scales)
        for (const void** p : {&table, &table_scale}) {
            if (*p == nullptr) continue;
            cudaPointerAttributes pa;
            if (cudaPointerGetAttributes(&pa, *p) != cudaSuccess) {
                cudaGetLastError();
                return ENGRAM_ERR_NO_UVA;
            }
            if (pa.type != cudaMemoryTypeHost || pa.devicePointer == nullptr)
                return ENGRAM_ERR_NO_UVA;
            *p = pa.devicePointer;
        }
    }

    engram_handle* h = new (std::nothrow) engram_handle();
    if (h == nullptr) return ENGRAM_ERR_OOM;
    std::memset(static_cast<void*>(h), 0, sizeof(*h));
    h->cfg = c;
    h->C = C;
    h->K = K;
    h->N = N;
    h->num_sms = sms;
    h->table = static_cast<const uint16_t*>(table);
    h->table_scale = static_cast<const uint8_t*>(table_scale);
    h->wkv = w->wkv;
    h->wkv_scale = w->wkv_scale;
    h->q = static_cast<const uint16_t*>(w->q_weight);
    h->k = static_cast<const uint16_t*>(w->k_weight);
    h->staged_T = -1;

    Workspace& ws = h->ws;
    ws.rows_alloc = (c.max_tokens + 255) / 256 * 256;
    const int64_t tdec = c.max_tokens < kMaxFusedT ? c.max_tokens : kMaxFusedT;
    ws.kv_tpitch = (tdec + 15) / 16 * 16;
    cudaError_t e = cudaSuccess;
    auto step = [&](cudaError_t r) {
        if (e == cudaSuccess) e = r;
    };
    step(dalloc(&h->d_row_offset, C * sizeof(int64_t), false));
    step(dalloc(&h->d_rows, C * sizeof(int64_t), false));
    step(dalloc(&ws.staged, ws.rows_alloc * K * 2, true));
    if (mx) {
        step(dalloc(&ws.staged_q, ws.rows_alloc * K, true));
        step(dalloc(&ws.staged_s, ws.rows_alloc * K / 32, true));
        // one 512-byte atom per 128 rows of each prefill tile and 128-byte k-block
        step(dalloc(&ws.wsf_atoms,
                    (N / prefill_bn(h)) * ((prefill_bn(h) + 127) / 128) * (K / 128) * 512, false));
    }
    // prefill path (also taken by small T when a decode column slice would
    // be too wide)
    step(dalloc(&ws.partials,
                ws.rows_alloc * c.hc_mult * 2 * (c.dim / prefill_bn(h)) *
                    sizeof(float4),
                true));
    step(dalloc(&ws.value, ws.rows_alloc * c.dim * 2, true));
    step(dalloc(&ws.gate, ws.rows_alloc * c.hc_mult * sizeof(float), true));
    // fused decode kernel workspace, sized for the largest T it serves
    h->fused = fused_layout(N, c.dim, c.hc_mult, sms);
    if (h->fused.ok) {
        step(dalloc(&ws.wpack, N * K * (mx ? 1 : 2), false));
        // gate-partial records: per copy [kv_tpitch][CTAs holding its keys] x 16 bytes
        step(dalloc(&ws.fpart, ws.kv_tpitch * (h->fused.grid + kMaxCopies) * 4 * sizeof(float),
                    true));
    }
    step(dalloc(&ws.fvalue, ws.kv_tpitch * c.dim * sizeof(float), true));
    step(dalloc(&ws.grid_bar, kFusedCounters * sizeof(unsigned long long), true));
    step(dalloc(&ws.qk, c.hc_mult * c.dim * sizeof(float), false));
    step(dalloc(&ws.err, sizeof(unsigned), true));
    if (e == cudaSuccess)
        e = cudaMemcpy(h->d_row_offset, w->row_offset, C * sizeof(int64_t), cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
        e = cudaMemcpy(h->d_rows, w->rows, C * sizeof(int64_t), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = launch_qk(h, 0);
    if (e == cudaSuccess) e = pack_weights(h, 0);
    if (e == cudaSuccess && mx) e = pack_scale_atoms(h, 0);
    if (e == cudaSuccess) e = gemm_setup_attributes();
    if (e == cudaSuccess) e = fused_setup_attributes();
    if (e == cudaSuccess) e = gate_setup_attributes();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        free_handle(h);
        return e == cudaErrorMemoryAllocation ? ENGRAM_ERR_OOM : ENGRAM_ERR_CUDA;
    }

    // token operand: bf16 rows, or their e4m3 codes for MXFP8
    const CUtensorMapDataType dt =
        mx ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int elem = mx ? 1 : 2;
    const void* act = mx ? static_cast<const void*>(ws.staged_q) : static_cast<const void*>(ws.staged);
    bool ok = make_map(&h->tm_w_n, h->wkv, dt, elem, K, N, prefill_bn(h)) &&
              make_map(&h->tm_w_half, h->wkv, dt, elem, K, N, prefill_bn(h) / 2) &&
              make_map(&h->tm_act_m, act, dt, elem, K, ws.rows_alloc, kBM);
    for (int i = 0; i < 16 && ok; ++i)
        ok = make_map(&h->tm_act_n[i], act, dt, elem, K, ws.rows_alloc, 16 * (i + 1));
    if (ok && mx) {
        const int bn = prefill_bn(h);
        const int atoms = (bn + 127) / 128;  // per tile and k-block
        ok = make_atom_map(&h->tm_sfa, ws.staged_s, ws.rows_alloc / kBM * (K / 128), 1) &&
             make_atom_map(&h->tm_sfb, ws.wsf_atoms, (N / bn) * (K / 128) * atoms, atoms);
    }
    if (!ok) {
        free_handle(h);
        return ENGRAM_ERR_CUDA;
    }
    h->gemm_pair_clusters = gemm_pair_capacity(h);
    *out = h;
    return ENGRAM_OK;
}

int engram_destroy(engram_t* h) {
    if (h == nullptr) return ENGRAM_OK;
    DeviceGuard guard(h->cfg.device);
    cudaDeviceSynchronize();
    free_handle(h);
    return ENGRAM_OK;
}

int engram_lookup(engram_t* h, const int32_t* hash_ids, int64_t ids_row_stride, int64_t T,
                  int background, cudaStream_t stream) {
    if (h == nullptr) return ENGRAM_ERR_INVALID_ARG;
    if (T < 0) return set_err(h, ENGRAM_ERR_INVALID_ARG);
    if (T > h->cfg.max_tokens) return set_err(h, ENGRAM_ERR_T_EXCEEDS_MAX);
    if (T == 0) {
        h->staged_T = 0;
        return set_err(h, ENGRAM_OK);
    }
    if (hash_ids == nullptr || ids_row_stride < h->C) return set_err(h, ENGRAM_ERR_INVALID_ARG);
    DeviceGuard guard(h->cfg.device);
    if (!guard.ok) return set_err(h, ENGRAM_ERR_CUDA);
    cudaError_t e = launch_gather(h, hash_ids, ids_row_stride, T, background != 0,
                                  h->cfg.wkv_format == ENGRAM_WKV_MXFP8, stream, false);
    if (e != cudaSuccess) return cuda_err(h, e);
    h->staged_T = T;
    return set_err(h, ENGRAM_OK);
}

int engram_forward(engram_t* h, const void* hidden, const int64_t hidden_strides[3],
                   const int32_t* hash_ids, int64_t ids_row_stride, const uint8_t* token_mask,
                   void* out, const int64_t out_strides[3], int64_t T, cudaStream_t stream) {
    if (h == nullptr) return ENGRAM_ERR_INVALID_ARG;
    if (T < 0) return set_err(h, ENGRAM_ERR_INVALID_ARG);
    if (T > h->cfg.max_tokens) return set_err(h, ENGRAM_ERR_T_EXCEEDS_MAX);
    if (T == 0) return set_err(h, ENGRAM_OK);
    const int64_t H = h->cfg.hc_mult, D = h->cfg.dim;
    int rc = check_view(hidden, hidden_strides);
    if (rc != ENGRAM_OK) return set_err(h, rc);
    rc = check_view(out, out_strides);
    if (rc != ENGRAM_OK) return set_err(h, rc);
    if (!rows_disjoint(out_strides, T, H, D)) return set_err(h, ENGRAM_ERR_INVALID_ARG);
    const bool same = hidden == out && hidden_strides[0] == out_strides[0] &&
                      hidden_strides[1] == out_strides[1];
    const int64_t ob = span_bytes(out_strides, T, H, D);
    if (!same && ranges_overlap(hidden, span_bytes(hidden_strides, T, H, D), out, ob))
        return set_err(h, ENGRAM_ERR_INVALID_ARG);
    if (hash_ids != nullptr && ids_row_stride < h->C) return set_err(h, ENGRAM_ERR_INVALID_ARG);
    // the ids and the mask are read while out is written: no overlap
    if ((hash_ids != nullptr &&
         ranges_overlap(out, ob, hash_ids, ((T - 1) * ids_row_stride + h->C) * 4)) ||
        (token_mask != nullptr && ranges_overlap(out, ob, token_mask, T)))
        return set_err(h, ENGRAM_ERR_INVALID_ARG);
    if (hash_ids == nullptr && h->staged_T != T) return set_err(h, ENGRAM_ERR_INVALID_ARG);

    DeviceGuard guard(h->cfg.device);
    if (!guard.ok) return set_err(h, ENGRAM_ERR_CUDA);
    const bool prof = h->profiling != 0;
    bool first = true;
    cudaError_t e = cudaSuccess;
    auto mark = [&](int i) {
        if (prof && e == cudaSuccess) e = cudaEventRecord(h->ev[i], stream);
    };
    if (fused_supported(h, T)) {
        // decode: one cooperative kernel, the gather included when ids are given
        h->ev_ran[0] = false;
        h->ev_ran[1] = true;
        h->ev_ran[2] = false;
        mark(0);
        mark(1);
        e = launch_decode_fused(h, hidden, hidden_strides, hash_ids, ids_row_stride, token_mask,
                                out, out_strides, T, stream, !prof);
        if (hash_ids != nullptr && e == cudaSuccess) h->staged_T = T;  // the kernel staged the rows
        mark(2);
        mark(3);
        h->last_path = 3;
        return cuda_err(h, e);
    }
    h->ev_ran[0] = hash_ids != nullptr;
    h->ev_ran[1] = h->ev_ran[2] = true;
    mark(0);
    if (hash_ids != nullptr) {
        e = launch_gather(h, hash_ids, ids_row_stride, T, false,
                          h->cfg.wkv_format == ENGRAM_WKV_MXFP8, stream, false);
        if (e != cudaSuccess) return cuda_err(h, e);
        h->staged_T = T;
        first = false;
    }
    mark(1);
    {
        if (e == cudaSuccess)
            e = launch_wkv_tokens_m(h, hidden, hidden_strides[0], hidden_strides[1], T, stream,
                                    !first && !prof);
        mark(2);
        if (e == cudaSuccess)
            e = launch_gate_from_partials(h, hidden, hidden_strides, token_mask, out, out_strides,
                                          T, stream, !prof);
        h->last_path = 2;
    }
    mark(3);
    return cuda_err(h, e);
}

int engram_debug_barrier_skew(engram_t* h, int64_t delta) {
    if (h == nullptr || delta < 0) return ENGRAM_ERR_INVALID_ARG;
    DeviceGuard guard(h->cfg.device);
    if (!guard.ok) return ENGRAM_ERR_CUDA;
    // the fused kernel's launch counter (the first of its four 64-bit counters)
    unsigned long long ctr = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&ctr, h->ws.grid_bar, sizeof(ctr), cudaMemcpyDeviceToHost);
    ctr += static_cast<unsigned long long>(delta);
    if (e == cudaSuccess) e = cudaMemcpy(h->ws.grid_bar, &ctr, sizeof(ctr), cudaMemcpyHostToDevice);
    return cuda_err(h, e);
}

int engram_wkv(engram_t* h, const int32_t* hash_ids, int64_t ids_row_stride, void* kv,
               int64_t kv_row_stride, int64_t T, cudaStream_t stream) {
    if (h == nullptr) return ENGRAM_ERR_INVALID_ARG;
    if (T < 0) return set_err(h, ENGRAM_ERR_INVALID_ARG);
    if (T > h->cfg.max_tokens) return set_err(h, ENGRAM_ERR_T_EXCEEDS_MAX);
    if (T == 0) return set_err(h, ENGRAM_OK);
    if (kv == nullptr || !aligned16(kv) || kv_row_stride < h->N || kv_row_stride % 8 != 0)
        return set_err(h, ENGRAM_ERR_INVALID_ARG);
    if (hash_ids != nullptr && ids_row_stride < h->C) return set_err(h, ENGRAM_ERR_INVALID_ARG);
    if (hash_ids == nullptr && h->staged_T != T) return set_err(h, ENGRAM_ERR_INVALID_ARG);
    if (!fused_supported(h, T)) return set_err(h, ENGRAM_ERR_UNSUPPORTED);
    DeviceGuard guard(h->cfg.device);
    if (!guard.ok) return set_err(h, ENGRAM_ERR_CUDA);
    // the decode kernel in kv mode: gather (when ids are given) and
    // projection, the gate and residual left out
    const cudaError_t e =
        launch_decode_fused(h, nullptr, nullptr, hash_ids, ids_row_stride, nullptr, nullptr,
                            nullptr, T, stream, h->profiling == 0, static_cast<uint16_t*>(kv),
                            kv_row_stride);
    if (hash_ids != nullptr && e == cudaSuccess) h->staged_T = T;
    h->last_path = 0;  // no gate or value of a forward to report
    return cuda_err(h, e);
}

int engram_debug_fused_plan(const engram_config* cfg, int64_t T, int32_t num_sms,
                            int64_t* out, int32_t n_out) {
    if (cfg == nullptr || out == nullptr || n_out < ENGRAM_FUSED_PLAN_FIELDS || num_sms < 1 ||
        T < 1 || cfg->dim <= 0 || cfg->hc_mult <= 0 || cfg->max_ngram_size < 2 ||
        cfg->n_heads < 1 || cfg->head_dim <= 0)
        return ENGRAM_ERR_INVALID_ARG;
    // the host planning of engram_create and engram_forward, on a handle
    // that holds only the configuration (no device is touched)
    engram_handle h;
    std::memset(static_cast<void*>(&h), 0, sizeof(h));
    h.cfg = *cfg;
    h.C = (cfg->max_ngram_size - 1) * cfg->n_heads;
    h.K = h.C * cfg->head_dim;
    h.N = cfg->dim * (cfg->hc_mult + 1);
    h.fused = fused_layout(h.N, cfg->dim, cfg->hc_mult, num_sms);
    const bool mx = cfg->wkv_format == ENGRAM_WKV_MXFP8;
    const FusedPlan p = fused_plan(&h, T);
    const FusedSmem m = fused_smem(h.fused, p, mx);
    const int64_t v[ENGRAM_FUSED_PLAN_FIELDS] = {
        fused_supported(&h, T) && m.ok ? 1 : 0, h.fused.grid, h.fused.max_width, p.mtiles,
        p.k_blocks, m.w_stages, m.x_stages, m.w_stage_bytes, m.x_stage_bytes, m.x_off,
        m.x_ring, m.qk_off, m.bar_off, kFusedSmemBytes, m.dual, p.Tn};
    for (int i = 0; i < ENGRAM_FUSED_PLAN_FIELDS; ++i) out[i] = v[i];
    return ENGRAM_OK;
}

int engram_forward_host(engram_t* h, const void* hidden_host, const int32_t* hash_ids_host,
                        const uint8_t* token_mask_host, void* out_host, int64_t T,
                        cudaStream_t stream) {
    if (h == nullptr) return ENGRAM_ERR_INVALID_ARG;
    if (T < 0) return set_err(h, ENGRAM_ERR_INVALID_ARG);
    if (T > h->cfg.max_tokens) return set_err(h, ENGRAM_ERR_T_EXCEEDS_MAX);
    if (T == 0) return set_err(h, ENGRAM_OK);
    if (hidden_host == nullptr || hash_ids_host == nullptr || out_host == nullptr)
        return set_err(h, ENGRAM_ERR_INVALID_ARG);
    DeviceGuard guard(h->cfg.device);
    if (!guard.ok) return set_err(h, ENGRAM_ERR_CUDA);
    const int64_t H = h->cfg.hc_mult, D = h->cfg.dim, C = h->C;
    Workspace& ws = h->ws;
    cudaError_t e = cudaSuccess;
    if (ws.host_hidden == nullptr) {
        e = dalloc(reinterpret_cast<uint16_t**>(&ws.host_hidden), ws.rows_alloc * H * D * 2, false);
        if (e == cudaSuccess) e = dalloc(&ws.host_ids, ws.rows_alloc * C * sizeof(int32_t), false);
        if (e == cudaSuccess) e = dalloc(&ws.host_mask, ws.rows_alloc, false);
        if (e != cudaSuccess) return cuda_err(h, e);
    }
    const size_t hb = static_cast<size_t>(T * H * D * 2);
    e = cudaMemcpyAsync(ws.host_hidden, hidden_host, hb, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(ws.host_ids, hash_ids_host, static_cast<size_t>(T * C * 4),
                            cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess && token_mask_host != nullptr)
        e = cudaMemcpyAsync(ws.host_mask, token_mask_host, static_cast<size_t>(T),
                            cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_err(h, e);
    const int64_t st[3] = {H * D, D, 1};
    int rc = engram_forward(h, ws.host_hidden, st, ws.host_ids, C,
                            token_mask_host != nullptr ? ws.host_mask : nullptr, ws.host_hidden, st,
                            T, stream);
    if (rc != ENGRAM_OK) return rc;
    e = cudaMemcpyAsync(out_host, ws.host_hidden, hb, cudaMemcpyDeviceToHost, stream);
    return cuda_err(h, e);
}

int engram_forward_host_pipelined(engram_t* h, const void* hidden_host,
                                  const int32_t* hash_ids_host, const uint8_t* token_mask_host,
                                  void* out_host, int64_t T, uint32_t flags, cudaStream_t stream) {
    if (h == nullptr) return ENGRAM_ERR_INVALID_ARG;
    if (T < 0 || (flags & ~ENGRAM_HOST_DEFER_OUTPUT) != 0u) return set_err(h, ENGRAM_ERR_INVALID_ARG);
    if (T > h->cfg.max_tokens) return set_err(h, ENGRAM_ERR_T_EXCEEDS_MAX);
    if (T == 0) return set_err(h, ENGRAM_OK);
    if (hidden_host == nullptr || hash_ids_host == nullptr || out_host == nullptr)
        return set_err(h, ENGRAM_ERR_INVALID_ARG);
    DeviceGuard guard(h->cfg.device);
    if (!guard.ok) return set_err(h, ENGRAM_ERR_CUDA);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) return cuda_err(h, e);
    if (cap != cudaStreamCaptureStatusNone)  // a graph holds one ordered sequence
        return engram_forward_host(h, hidden_host, hash_ids_host, token_mask_host, out_host, T,
                                   stream);
    const int64_t H = h->cfg.hc_mult, D = h->cfg.dim, C = h->C;
    Workspace& ws = h->ws;
    if (h->pipe_in == nullptr) {
        for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
            e = dalloc(reinterpret_cast<uint16_t**>(&ws.pipe_hidden[b]), ws.rows_alloc * H * D * 2,
                       false);
            if (e == cudaSuccess) e = dalloc(&ws.pipe_ids[b], ws.rows_alloc * C * sizeof(int32_t), false);
            if (e == cudaSuccess) e = dalloc(&ws.pipe_mask[b], ws.rows_alloc, false);
            for (cudaEvent_t* ev : {&h->pipe_ev_in[b], &h->pipe_ev_fwd[b], &h->pipe_ev_out[b]})
                if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        }
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->pipe_out, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->pipe_in, cudaStreamNonBlocking);
        if (e != cudaSuccess) return cuda_err(h, e);  // (freed with the handle)
    }
    const int b = static_cast<int>(h->pipe_calls & 1u);
    const size_t hb = static_cast<size_t>(T * H * D * 2);
    // inputs into slot b once the call two back has copied its output out of
    // it (that copy followed its forward, the slot's last reader)
    if (h->pipe_calls >= 2) e = cudaStreamWaitEvent(h->pipe_in, h->pipe_ev_out[b], 0);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(ws.pipe_hidden[b], hidden_host, hb, cudaMemcpyHostToDevice, h->pipe_in);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(ws.pipe_ids[b], hash_ids_host, static_cast<size_t>(T * C * 4),
                            cudaMemcpyHostToDevice, h->pipe_in);
    if (e == cudaSuccess && token_mask_host != nullptr)
        e = cudaMemcpyAsync(ws.pipe_mask[b], token_mask_host, static_cast<size_t>(T),
                            cudaMemcpyHostToDevice, h->pipe_in);
    if (e == cudaSuccess) e = cudaEventRecord(h->pipe_ev_in[b], h->pipe_in);
    // the forward on the caller's stream, in place in slot b
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, h->pipe_ev_in[b], 0);
    if (e != cudaSuccess) return cuda_err(h, e);
    const int64_t st[3] = {H * D, D, 1};
    const int rc = engram_forward(h, ws.pipe_hidden[b], st, ws.pipe_ids[b], C,
                                  token_mask_host != nullptr ? ws.pipe_mask[b] : nullptr,
                                  ws.pipe_hidden[b], st, T, stream);
    if (rc != ENGRAM_OK) return rc;
    // the output copy on the output stream; the caller's stream waits for it
    e = cudaEventRecord(h->pipe_ev_fwd[b], stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->pipe_out, h->pipe_ev_fwd[b], 0);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(out_host, ws.pipe_hidden[b], hb, cudaMemcpyDeviceToHost, h->pipe_out);
    if (e == cudaSuccess) e = cudaEventRecord(h->pipe_ev_out[b], h->pipe_out);
    // the caller's stream waits for this output copy, or (deferred) for the
    // previous call's, which the forward just run has long overtaken
    if (e == cudaSuccess) {
        if (!(flags & ENGRAM_HOST_DEFER_OUTPUT))
            e = cudaStreamWaitEvent(stream, h->pipe_ev_out[b], 0);
        else if (h->pipe_calls >= 1)
            e = cudaStreamWaitEvent(stream, h->pipe_ev_out[b ^ 1], 0);
    }
    if (e == cudaSuccess) ++h->pipe_calls;
    return cuda_err(h, e);
}

int engram_forward_host_flush(engram_t* h, cudaStream_t stream) {
    if (h == nullptr) return ENGRAM_ERR_INVALID_ARG;
    if (h->pipe_calls == 0) return set_err(h, ENGRAM_OK);
    DeviceGuard guard(h->cfg.device);
    if (!guard.ok) return set_err(h, ENGRAM_ERR_CUDA);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cap);
    if (e == cudaSuccess && cap == cudaStreamCaptureStatusNone)
        e = cudaStreamWaitEvent(stream, h->pipe_ev_out[(h->pipe_calls - 1) & 1u], 0);
    return cuda_err(h, e);
}

int engram_last_error(engram_t* h, int sync) {
    if (h == nullptr) return ENGRAM_ERR_INVALID_ARG;
    if (sync) {
        uint32_t bits = 0;
        int rc = engram_device_error(h, &bits, 1);
        if (rc != ENGRAM_OK) return rc;
        if (bits != 0) return ENGRAM_ERR_DEVICE;
    }
    return h->last_error;
}

int engram_device_error(engram_t* h, uint32_t* bits, int clear) {
    if (h == nullptr || bits == nullptr) return ENGRAM_ERR_INVALID_ARG;
    DeviceGuard guard(h->cfg.device);
    if (!guard.ok) return ENGRAM_ERR_CUDA;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(bits, h->ws.err, sizeof(unsigned), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && clear) e = cudaMemset(h->ws.err, 0, sizeof(unsigned));
    if (e == cudaSuccess && (*bits & ENGRAM_DEVERR_TIMEOUT)) {
        // an unwound launch can leave the grid barrier's arrival count
        // short: start it again from zero
        e = cudaMemset(h->ws.grid_bar, 0, kFusedCounters * sizeof(unsigned long long));
    }
    if (e != cudaSuccess) return ENGRAM_ERR_CUDA;
    return ENGRAM_OK;
}

int engram_debug_intermediates(engram_t* h, float* gate, float* value, int64_t T,
                               cudaStream_t stream) {
    if (h == nullptr || T < 0 || T > h->cfg.max_tokens) return ENGRAM_ERR_INVALID_ARG;
    if (T == 0) return ENGRAM_OK;
    DeviceGuard guard(h->cfg.device);
    if (!guard.ok) return ENGRAM_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    if (gate != nullptr)
        e = cudaMemcpyAsync(gate, h->ws.gate, T * h->cfg.hc_mult * sizeof(float),
                            cudaMemcpyDeviceToDevice, stream);
    if (e == cudaSuccess && value != nullptr) {
        if (h->last_path == 0)
            return ENGRAM_ERR_INVALID_ARG;
        e = h->last_path == 3 ? launch_fused_debug_value(h, value, T, stream)
                              : launch_debug_value(h, value, T, stream);
    }
    return e == cudaSuccess ? ENGRAM_OK : ENGRAM_ERR_CUDA;
}

int engram_debug_staged_rows(engram_t* h, void* rows, int64_t T, cudaStream_t stream) {
    if (h == nullptr || rows == nullptr || T < 0 || T > h->cfg.max_tokens)
        return ENGRAM_ERR_INVALID_ARG;
    if (T == 0) return ENGRAM_OK;
    DeviceGuard guard(h->cfg.device);
    if (!guard.ok) return ENGRAM_ERR_CUDA;
    cudaError_t e = cudaMemcpyAsync(rows, h->ws.staged, T * h->K * 2, cudaMemcpyDeviceToDevice,
                                    stream);
    return e == cudaSuccess ? ENGRAM_OK : ENGRAM_ERR_CUDA;
}

int engram_debug_staged_mx(engram_t* h, uint8_t* codes, uint8_t* scales, int64_t T,
                           cudaStream_t stream) {
    if (h == nullptr || T < 0 || T > h->cfg.max_tokens) return ENGRAM_ERR_INVALID_ARG;
    if (h->cfg.wkv_format != ENGRAM_WKV_MXFP8) return ENGRAM_ERR_INVALID_ARG;
    if (T == 0) return ENGRAM_OK;
    DeviceGuard guard(h->cfg.device);
    if (!guard.ok) return ENGRAM_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    if (codes != nullptr)
        e = cudaMemcpyAsync(codes, h->ws.staged_q, T * h->K, cudaMemcpyDeviceToDevice, stream);
    if (e == cudaSuccess && scales != nullptr) e = launch_unpack_scales(h, scales, T, stream);
    return e == cudaSuccess ? ENGRAM_OK : ENGRAM_ERR_CUDA;
}

int engram_debug_keep_value(engram_t* h, int enable) {
    if (h == nullptr) return ENGRAM_ERR_INVALID_ARG;
    h->keep_value = enable != 0;
    return set_err(h, ENGRAM_OK);
}

int engram_profile_enable(engram_t* h, int enable) {
    if (h == nullptr) return ENGRAM_ERR_INVALID_ARG;
    DeviceGuard guard(h->cfg.device);
    if (!guard.ok) return set_err(h, ENGRAM_ERR_CUDA);
    if (enable && h->ev[0] == nullptr) {
        for (cudaEvent_t& ev : h->ev) {
            if (cudaEventCreate(&ev) == cudaSuccess) continue;
            ev = nullptr;
            for (cudaEvent_t& made : h->ev) {  // all or none
                if (made != nullptr) cudaEventDestroy(made);
                made = nullptr;
            }
            return set_err(h, ENGRAM_ERR_CUDA);
        }
    }
    h->profiling = enable != 0;
    return set_err(h, ENGRAM_OK);
}

int engram_profile_read(engram_t* h, float ms[3]) {
    if (h == nullptr || ms == nullptr || h->ev[0] == nullptr) return ENGRAM_ERR_INVALID_ARG;
    DeviceGuard guard(h->cfg.device);
    if (!guard.ok) return ENGRAM_ERR_CUDA;
    if (cudaEventSynchronize(h->ev[3]) != cudaSuccess) return set_err(h, ENGRAM_ERR_CUDA);
    for (int i = 0; i < 3; ++i) {
        ms[i] = 0.f;
        if (h->ev_ran[i] && cudaEventElapsedTime(&ms[i], h->ev[i], h->ev[i + 1]) != cudaSuccess)
            return set_err(h, ENGRAM_ERR_CUDA);
    }
    return set_err(h, ENGRAM_OK);
}

}  // extern "C"
