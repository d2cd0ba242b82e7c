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
constexpr int kBNPrefill = 256;   // kv columns per prefill tile, bf16 wkv
constexpr int kBNPrefillMx = 128; // kv columns per prefill tile, MXFP8 wkv (TMEM holds the
                                  // two accumulators plus a scale-factor slot per stage)
constexpr int kBNPrefillMxWide = 224;  // the same when it divides dim (2 x 224 + 4 x 16 = 512)
constexpr int kKBlockBytes = 128; // bytes of K per pipeline stage (one swizzle row)
constexpr int kGemmSmemBytes = 192 * 1024 + 2048;  // > half an SM: one CTA per SM
constexpr int kFusedSmemBytes = 225 * 1024;       // fused decode kernel
constexpr int kMaxCopies = 4;                     // largest hc_mult
constexpr int kMaxFusedT = 256;                   // largest T of the fused decode kernel
constexpr int kMaxFusedSlice = 256;               // widest column slice of one CTA (MMA N)
constexpr int kMaxFusedTMx = 128;                 // largest T of the fused kernel, MXFP8 wkv
constexpr int kFusedCounters = 4;                 // 64-bit counters of the fused kernel

// MXFP8 scale-factor atoms: the E8M0 scales of 128 rows x 128 k (4 scales
// per row) as the 512-byte image tcgen05.cp .32x128b.warpx4 copies into
// TMEM: byte 16*i + 4*j + b holds the scale of row 32*j + i, k-block b.
// A [rows, K] operand's atoms are stored [rows/128][K/128][512].
__host__ __device__ inline int64_t sf_atom_offset(int64_t row, int64_t k32, int64_t kblocks128) {
    return ((row >> 7) * kblocks128 + (k32 >> 2)) * 512 + (row & 31) * 16 +
           ((row >> 5) & 3) * 4 + (k32 & 3);
}

struct Workspace {
    // staged gather output (Engram.staged_rows): bf16 [rows_alloc, K]
    uint16_t* staged = nullptr;
    int64_t rows_alloc = 0;  // max_tokens rounded up to 256
    // MXFP8 activations: e4m3 codes [rows_alloc, K] and their E8M0 scales
    // as atoms [rows_alloc/128][K/128][512]
    uint8_t* staged_q = nullptr;
    uint8_t* staged_s = nullptr;
    // tokens padded to 16 up to the fused kernel's largest T
    int64_t kv_tpitch = 0;
    // prefill path: fp32 (sum key^2, sum hidden*q*k*key) per key tile
    // [rows_alloc][H][D/BN] and the bf16 value [rows_alloc][D]
    float4* partials = nullptr;  // prefill: (sum hidden^2, sum key^2, sum h*q*k*key, -)
    uint16_t* value = nullptr;
    // fp32 gate of the last forward [rows_alloc][H]
    float* gate = nullptr;
    // fp32 q*k [H, D]
    float* qk = nullptr;
    // MXFP8 weight scales as atoms [N/128][K/128][512] (prefill B operand)
    uint8_t* wsf_atoms = nullptr;
    // sticky device error word
    unsigned* err = nullptr;
    // fused decode kernel: wkv packed k-block-major (128 bytes of k per row
    // and block) as swizzled shared-memory images, each CTA's columns
    // consecutive; gate-partial records; the fp32 value (validation only);
    // the kernel's counters (a launch counter and three grid barriers)
    uint8_t* wpack = nullptr;
    float* fpart = nullptr;     // records: per hc copy [kv_tpitch][CTAs covering it][4]
    float* fvalue = nullptr;    // [kv_tpitch][D]
    unsigned* grid_bar = nullptr;  // kFusedCounters 64-bit counters of the fused kernel
    // host path staging (engram_forward_host)
    void* host_hidden = nullptr;
    int32_t* host_ids = nullptr;
    uint8_t* host_mask = nullptr;
    // engram_forward_host_pipelined: two slots used in turn
    void* pipe_hidden[2] = {nullptr, nullptr};
    int32_t* pipe_ids[2] = {nullptr, nullptr};
    uint8_t* pipe_mask[2] = {nullptr, nullptr};
};

// Column ownership of the fused decode kernel: N = D*(H+1) columns in
// 16-column granules; CTA c owns NG-split granules [g0, g1), of which the
// first (VG-split) ones are value columns and the rest a run of key columns
// (first key granule = first_granule(c, NG) - first_granule(c, VG)).
struct FusedLayout {
    int grid, NG, VG, max_width;
    int cf[kMaxCopies], nh[kMaxCopies];  // first CTA and CTA count holding each copy's keys
    bool ok;
};

struct FusedPlan {
    int Tn, mtiles, k_blocks;
};

// Shared-memory plan of one fused launch (byte offsets from the 1024-byte
// aligned base): weight ring | token ring | q*k slice | barriers.
struct FusedSmem {
    uint32_t x_bytes, x_stage_bytes, w_stage_bytes, x_ring, x_off, qk_off, bar_off;
    int x_stages, w_stages, dual;
    bool ok;  // at least two weight stages fit
};

}  // namespace engram

struct engram_handle {
    engram_config cfg;
    int64_t C, K, N;
    int num_sms;
    // borrowed weights
    const uint16_t* table;        // bf16 rows, or e4m3 codes of an fp8 table
    const uint8_t* table_scale;   // fp8 table: ue8m0 [rows][E/32]; null for bf16
    const void* wkv;
    const uint8_t* wkv_scale;
    const uint16_t* q;
    const uint16_t* k;
    int64_t* d_row_offset;
    int64_t* d_rows;
    engram::Workspace ws;
    // TMA descriptors
    CUtensorMap tm_w_n;        // wkv, prefill B operand (box BN rows x 128 bytes)
    CUtensorMap tm_w_half;     // the same, box BN/2 rows (a CTA's half in a CTA-pair GEMM)
    CUtensorMap tm_sfa;        // MXFP8 scale atoms of the staged rows, rows of 512 bytes, box 1 row
    CUtensorMap tm_sfb;        // MXFP8 scale atoms of wkv, box = one prefill tile's atoms
    int gemm_pair_clusters;    // CTA-pair GEMM clusters that fit at once (0: single CTAs)
    CUtensorMap tm_act_m;      // staged rows (bf16, or e4m3 codes), box 128 rows x 128 bytes
    CUtensorMap tm_act_n[16];  // the same, box 16 * (i + 1) rows (the fused kernel's tile)
    engram::FusedLayout fused;
    int keep_value;  // validation: the fused kernel also stores the fp32 value
    // last lookup
    int64_t staged_T;
    int last_error;
    int last_path;  // 0 = none, 2 = prefill kernels, 3 = fused decode kernel
    // measurement hook
    int profiling;
    cudaEvent_t ev[4];
    bool ev_ran[3];
    // engram_forward_host_pipelined: input and output copy streams, and per
    // slot the events "inputs copied", "forward done", "output copied"
    cudaStream_t pipe_in, pipe_out;
    cudaEvent_t pipe_ev_in[2], pipe_ev_fwd[2], pipe_ev_out[2];
    uint64_t pipe_calls;
};

namespace engram {

// gather.cu
cudaError_t launch_gather(const engram_handle* h, const int32_t* ids, int64_t ids_stride,
                          int64_t T, bool background, bool quantize, cudaStream_t s, bool pdl);

// wkv_gemm.cu
cudaError_t launch_wkv_tokens_m(const engram_handle* h, const void* hidden, int64_t hs_t,
                                int64_t hs_h, int64_t T, cudaStream_t s, bool pdl);
cudaError_t gemm_setup_attributes();
int prefill_bn(const engram_handle* h);  // kv columns per prefill tile
int gemm_pair_capacity(const engram_handle* h);
cudaError_t pack_scale_atoms(const engram_handle* h, cudaStream_t s);
cudaError_t launch_unpack_scales(const engram_handle* h, uint8_t* out, int64_t T, cudaStream_t s);

// decode_fused.cu
FusedLayout fused_layout(int64_t N, int64_t D, int64_t H, int num_sms);
FusedPlan fused_plan(const engram_handle* h, int64_t T);
FusedSmem fused_smem(const FusedLayout& L, const FusedPlan& p, bool mx);
bool fused_supported(const engram_handle* h, int64_t T);
cudaError_t fused_setup_attributes();
cudaError_t gate_setup_attributes();
cudaError_t pack_weights(const engram_handle* h, cudaStream_t s);
cudaError_t launch_fused_debug_value(const engram_handle* h, float* value, int64_t T,
                                     cudaStream_t s);
// ids == nullptr: the rows were staged by engram_lookup
cudaError_t launch_decode_fused(engram_handle* h, const void* hidden, const int64_t* hs,
                                const int32_t* ids, int64_t ids_stride, const uint8_t* mask,
                                void* out, const int64_t* os, int64_t T, cudaStream_t s,
                                bool pdl, uint16_t* kv = nullptr, int64_t kv_ld = 0);

// gate.cu
cudaError_t launch_gate_from_partials(const engram_handle* h, const void* hidden,
                                      const int64_t* hs, const uint8_t* mask, void* out,
                                      const int64_t* os, int64_t T, cudaStream_t s, bool pdl);
cudaError_t launch_debug_value(const engram_handle* h, float* value, int64_t T, cudaStream_t s);
cudaError_t launch_qk(const engram_handle* h, cudaStream_t s);

}  // namespace engram
