// Hash-row gather (ParallelEngramEmbedding.lookup feeding Engram.staged_rows,
// "vllm.models.deepseek_v4_1.common.engram"):
//   staged[t, c*E + j] = table[row_offset[c] + ids[t, c], j]
// One thread moves one 16-byte chunk; the E/8 threads of a row are
// consecutive lanes, so every 128-byte row is one fully used request.  Each
// thread keeps kUnroll independent row reads in flight to cover the
// latency of random rows in HBM or, for an offloaded table, in host memory
// across the host link.  The grid is capped at a few CTAs per SM (half the
// SMs for a background lookup) that loop over the chunks: the table spans
// far more memory than the TLBs map, as the lookup's page points out.
// Optionally the same pass emits the MXFP8 form of the rows: e4m3
// codes and one E8M0 scale per 32 consecutive k (smallest power of two that
// keeps the block maximum within 448; round-to-nearest-even, saturating),
// the scales stored as the tcgen05 scale-factor atoms the GEMM copies.
// An fp8 table (e4m3 rows, one ue8m0 scale per 32 elements, class
// ParallelEngramEmbedding) is dequantized to bf16 on the way: a thread reads
// 8 code bytes and the row's scale byte for its 16-byte chunk.
#include "internal.h"
#include "mxfp8.cuh"
#include "ptx.cuh"

namespace engram {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kUnroll = 4;

struct GatherArgs {
    const uint16_t* table;     // bf16 rows, or (fp8) e4m3 codes [rows][E]
    const uint8_t* tscale;     // fp8 table: ue8m0 [rows][E/32]; else null
    const int64_t* row_offset;
    const int64_t* rows;
    const int32_t* ids;
    int64_t ids_stride;
    uint16_t* staged;  // [T, K]
    uint8_t* codes;    // [T, K]                     (quantize only)
    uint8_t* scales;   // atoms [T/128][K/128][512]  (quantize only)
    int64_t n_chunks;  // T * C * cpr
    int C, E, K, cpr_shift;
    unsigned* err;
};

template <bool kQuant>
__global__ void __launch_bounds__(kGatherThreads) gather_rows_kernel(const GatherArgs a) {
    pdl_wait();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kGatherThreads;
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = static_cast<int64_t>(blockIdx.x) * kGatherThreads + (threadIdx.x & ~31);
    const int cpr_mask = (1 << a.cpr_shift) - 1;
    unsigned bad = 0;
    // The loop bound is warp-uniform so every lane reaches the shuffles.
    for (int64_t base = warp0; base < a.n_chunks; base += stride * kUnroll) {
        uint4 v[kUnroll];
        int64_t dst[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t g = base + lane + u * stride;
            v[u] = make_uint4(0u, 0u, 0u, 0u);
            dst[u] = -1;
            if (g < a.n_chunks) {
                const int64_t r = g >> a.cpr_shift;  // (t, c) row
                const int j = static_cast<int>(g & cpr_mask);
                const int64_t t = r / a.C;
                const int c = static_cast<int>(r - t * a.C);
                const int64_t id = a.ids[t * a.ids_stride + c];
                dst[u] = r * a.E + j * 8;
                if (id >= 0 && id < __ldg(a.rows + c)) {
                    const int64_t row = __ldg(a.row_offset + c) + id;
                    if (a.tscale == nullptr) {
                        v[u] = ld_stream_v4(a.table + row * a.E + j * 8);
                    } else {
                        const uint8_t* cp = reinterpret_cast<const uint8_t*>(a.table) + row * a.E + j * 8;
                        v[u] = dequant8(__ldg(reinterpret_cast<const uint2*>(cp)),
                                        __ldg(a.tscale + row * (a.E >> 5) + (j >> 2)));
                    }
                } else {
                    bad = 1;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (dst[u] >= 0) st_v4(a.staged + dst[u], v[u]);
            if constexpr (kQuant) {
                // 4 consecutive lanes hold one 32-element block.
                uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                uint32_t m = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    m = max(m, w[i] & 0x7FFFu);
                    m = max(m, (w[i] >> 16) & 0x7FFFu);
                }
                m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
                m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
                const int e = mx_scale_exponent(__uint_as_float(m << 16));
                const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
                if (dst[u] >= 0) {
                    *reinterpret_cast<uint2*>(a.codes + dst[u]) =
                        make_uint2(mx_codes4(w[0], w[1], inv), mx_codes4(w[2], w[3], inv));
                    if ((lane & 3) == 0) {
                        const int64_t t = dst[u] / a.K;
                        a.scales[sf_atom_offset(t, (dst[u] - t * a.K) >> 5, a.K >> 7)] =
                            static_cast<uint8_t>(e + 127);
                    }
                }
            }
        }
    }
    if (bad) atomicOr(a.err, ENGRAM_DEVERR_BAD_HASH_ID);
    pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_gather(const engram_handle* h, const int32_t* ids, int64_t ids_stride,
                          int64_t T, bool background, bool quantize, cudaStream_t s, bool pdl) {
    GatherArgs a;
    a.table = h->table;
    a.tscale = h->table_scale;
    a.row_offset = h->d_row_offset;
    a.rows = h->d_rows;
    a.ids = ids;
    a.ids_stride = ids_stride;
    a.staged = h->ws.staged;
    a.codes = h->ws.staged_q;
    a.scales = h->ws.staged_s;
    a.C = static_cast<int>(h->C);
    a.E = static_cast<int>(h->cfg.head_dim);
    a.K = static_cast<int>(h->K);
    int cpr = a.E / 8, shift = 0;
    while ((1 << shift) < cpr) ++shift;
    a.cpr_shift = shift;
    a.n_chunks = T * h->C * cpr;
    a.err = h->ws.err;

    const int64_t per_block = static_cast<int64_t>(kGatherThreads) * kUnroll;
    int64_t blocks = (a.n_chunks + per_block - 1) / per_block;
    const int64_t cap = background ? (h->num_sms / 2 > 0 ? h->num_sms / 2 : 1)
                                   : static_cast<int64_t>(h->num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kGatherThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (quantize) return cudaLaunchKernelEx(&cfg, gather_rows_kernel<true>, a);
    return cudaLaunchKernelEx(&cfg, gather_rows_kernel<false>, a);
}

}  // namespace engram
