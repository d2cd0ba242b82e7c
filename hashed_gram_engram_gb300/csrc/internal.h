// Internal declarations shared by the library's translation units: the
// handle, the workspace layout, and the kernel launchers.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "engram.h"

namespace engram {

// wkv GEMM tiling.
constexpr int kBM = 128;          // MMA M: rows of the TMEM accumulator
constexpr int kBNPrefill = 256;   // kv columns per tile when tokens are the M side
constexpr int kKBlockBytes = 128; // bytes of K per pipeline stage (one swizzle row)
constexpr int kGemmSmemBytes = 192 * 1024 + 2048;  // > half an SM: one CTA per SM
constexpr int kFusedSmemBytes = 225 * 1024;       // fused decode kernel
constexpr int kMaxFusedT = 256;                   // largest T of the fused decode kernel
constexpr int kMaxFusedSlice = 256;               // widest column slice of one CTA (MMA N)

struct Workspace {
    // staged gather output (Engram.staged_rows): bf16 [rows_alloc, K]
    uint16_t* staged = nullptr;
    int64_t rows_alloc = 0;  // max_tokens rounded up to 256
    // MXFP8 activations: e4m3 codes [rows_alloc, K], E8M0 scales [rows_alloc, K/32]
    uint8_t* staged_q = nullptr;
    uint8_t* staged_s = nullptr;
    // tokens padded to 16 up to the fused kernel's largest T
    int64_t kv_tpitch = 0;
    // prefill path: fp32 (sum key^2, sum hidden*q*k*key) per 256-column key
    // tile [rows_alloc][H][D/256] and the bf16 value [rows_alloc][D]
    float2* partials = nullptr;
    uint16_t* value = nullptr;
    // fp32 gate of the last forward [rows_alloc][H]
    float* gate = nullptr;
    // fp32 q*k [H, D]
    float* qk = nullptr;
    // MXFP8 weight scales expanded per row: [N][K/32] bytes
    uint8_t* wscale_rows = nullptr;
    // sticky device error word
    unsigned* err = nullptr;
    // fused decode kernel: wkv packed k-block-major as swizzled shared-memory
    // images, per-(token, CTA) gate partial sums, the fp32 value, the
    // grid-barrier counter
    uint16_t* wpack = nullptr;
    float* fpart = nullptr;     // [kv_tpitch][num_sms][8]
    float* fvalue = nullptr;    // [kv_tpitch][D]
    unsigned* grid_bar = nullptr;  // two {count, generation} grid barriers of the fused kernel
    // host path staging (engram_forward_host)
    void* host_hidden = nullptr;
    int32_t* host_ids = nullptr;
    uint8_t* host_mask = nullptr;
};

struct FusedPlan {
    int Tn, mtiles, granules, k_blocks, grid, max_width;
};

}  // namespace engram

struct engram_handle {
    engram_config cfg;
    int64_t C, K, N;
    int num_sms;
    // borrowed weights
    const uint16_t* table;
    const void* wkv;
    const uint8_t* wkv_scale;
    const uint16_t* q;
    const uint16_t* k;
    int64_t* d_row_offset;
    int64_t* d_rows;
    engram::Workspace ws;
    // TMA descriptors
    CUtensorMap tm_w_n;                 // wkv as the N-side operand (box 256 rows)
    CUtensorMap tm_act_m;               // staged rows as the M-side operand (box 128 rows)
    CUtensorMap tm_act_n[16];           // staged rows as the N-side operand (box 16..256 rows)
    CUtensorMap tm_sfw;                 // MXFP8 weight scales per row
    CUtensorMap tm_sfa_n[16];           // MXFP8 activation scales per row (N side)
    // last lookup
    int64_t staged_T;
    int last_error;
    int last_path;  // 0 = none, 2 = prefill kernels, 3 = fused decode kernel
    // measurement hook
    int profiling;
    cudaEvent_t ev[4];
    bool ev_ran[3];
};

namespace engram {

// gather.cu
cudaError_t launch_gather(const engram_handle* h, const int32_t* ids, int64_t ids_stride,
                          int64_t T, bool background, bool quantize, cudaStream_t s, bool pdl);

// wkv_gemm.cu
cudaError_t launch_wkv_tokens_m(const engram_handle* h, const void* hidden, int64_t hs_t,
                                int64_t hs_h, int64_t T, cudaStream_t s, bool pdl);
cudaError_t gemm_setup_attributes();

// decode_fused.cu
FusedPlan fused_plan(const engram_handle* h, int64_t T);
bool fused_supported(const engram_handle* h, int64_t T);
cudaError_t fused_setup_attributes();
cudaError_t pack_weights(const engram_handle* h, cudaStream_t s);
cudaError_t launch_fused_debug_value(const engram_handle* h, float* value, int64_t T,
                                     cudaStream_t s);
// ids == nullptr: the rows were staged by engram_lookup
cudaError_t launch_decode_fused(engram_handle* h, const void* hidden, const int64_t* hs,
                                const int32_t* ids, int64_t ids_stride, const uint8_t* mask,
                                void* out, const int64_t* os, int64_t T, cudaStream_t s);

// gate.cu
cudaError_t launch_gate_from_partials(const engram_handle* h, const void* hidden,
                                      const int64_t* hs, const uint8_t* mask, void* out,
                                      const int64_t* os, int64_t T, cudaStream_t s, bool pdl);
cudaError_t launch_debug_value(const engram_handle* h, float* value, int64_t T, cudaStream_t s);
cudaError_t launch_qk(const engram_handle* h, cudaStream_t s);

}  // namespace engram
