// The whole Engram forward of a decode step (T <= 256; MXFP8 wkv T <= 128)
// in one cooperative, persistent kernel, one CTA per SM.  Engram.forward
// ("vllm.models.deepseek_v4_1.common.engram") defines the layer; the gate
// arithmetic is that of _engram_gate_finish_kernel with one rank, split over
// dim the way _engram_gate_partials_kernel splits it over ranks
// ("vllm.models.deepseek_v41.amd.engram").
//
// Column ownership.  The N = D*(H+1) kv columns are cut into 16-column
// granules; CTA c owns a balanced share of them, made of a few VALUE
// granules (dims [v0, v0 + vlen) of the shared value) followed by a run of
// KEY columns [k0, k0 + klen) (which may straddle two hc copies).  wkv is
// packed at create time so that each CTA's rows are consecutive.  Because a
// CTA holds the value of its dims for every token, it finishes those output
// dims itself: the only data that crosses SMs after the projection are the
// gate partial sums.
//
// Roles (224 threads): warp 0 streams the CTA's weight slice through a deep
// ring of k-block stages from the first instant (bulk copies of >= 16 KB
// keep enough bytes in flight for full HBM bandwidth); warp 1 owns TMEM and
// issues the tcgen05 MMAs (tokens on M, the slice on N, fp32 accumulators
// in TMEM) -- for bf16 with T <= 128 it takes the even k-blocks and warp 6
// the odd ones into a second accumulator (one thread's issue loop cannot
// keep the tensor pipe busy on these small MMAs), the two summed when read;
// warps 2-5 gather, then run the epilogue and the residual (TMEM lane
// quarter = warp % 4).  The token tiles come through their own ring of TMA
// tensor copies (one box of the staged rows per k-block, 128-byte swizzled
// by the copy engine), issued by one thread of warp 2: per-thread cp.async
// from a few warps could not keep enough bytes in flight.
//
//   gather   each CTA copies ~1/grid of the T x C hash rows into the
//            staged buffer (an fp8 table's rows dequantized to bf16 on the
//            way; MXFP8 wkv: the rows also quantised into e4m3 codes and
//            scales); grid barrier 1; then every CTA loads the token tiles
//            of every k-block from the staged rows.  Rows staged by
//            engram_lookup skip the gather;
//   epilogue thread = token: for the key columns it sums hidden^2, key^2
//            and hidden*q*k*key per hc copy into a record per (copy, token,
//            CTA).  With one token tile and at most 48 value dims it also
//            loads the residual's operands now (the value from TMEM, hidden
//            at its value dims); grid barrier 2;
//   gates    CTA c reduces the records of rows (token, copy) = c, c + grid,
//            ... (one warp per row, a fixed summation order: runs are
//            bit-identical) and publishes the gates; grid barrier 3;
//   residual every CTA writes hidden + gate * value for its own value dims
//            (masked tokens keep hidden's bits), the value read straight
//            from TMEM (or from the registers loaded before barrier 2).
//
// Template parameters: the wkv format (bf16 / MXFP8) and the table format
// (bf16 / e4m3 with ue8m0 scales), so that neither path pays for the
// other's code.
//
// The launch is programmatic-dependent: the next launch may start once every
// CTA has begun; before griddepcontrol.wait a CTA only sets up and starts the
// weight stream (wkv is never written by a kernel).
//
// MXFP8 wkv (T <= 128): the gather also quantises the rows (e4m3 codes and
// E8M0 scales per 32 k); the MMAs are kind::mxf8f6f4 block_scale and the
// scale factors sit in TMEM next to the accumulator.  A slice starts on any
// 16-column boundary, so the epilogue warps write the scale words into TMEM
// (tcgen05.st) rather than copying 128-row atoms: the weights' at kernel
// start, the tokens' after the gather.  Scale cell layout (scale_vec::1X):
// the scale of A row r for k-block b is byte b of lane r, column
// sfa + r / 32; that of B row n is byte b of lane n % 32, column sfb + n / 32.
//
// Grid barriers: counters that only grow.  Each launch reads its epoch e
// from a launch counter at start (CTA 0 advances it at the very end); a
// CTA arrives with a posted release add and waits until the counter reaches
// e * grid.  No reset, so a captured launch replays.  Every wait is bounded.
#include <cuda_bf16.h>

#include "internal.h"
#include "mxfp8.cuh"
#include "ptx.cuh"

namespace engram {
namespace {

constexpr int kThreads = 224;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxWStages = 12;
constexpr int kMaxXStages = 12;
constexpr uint32_t kXRingTarget = 96 * 1024;  // bytes of token stages
constexpr int kKeyChunks = kMaxFusedSlice / 16;  // 16-column chunks of a slice
constexpr uint32_t kTmemCols = 512;

struct FusedArgs {
    int T, Tn, D, H, C, E, N, K;
    int mtiles, NG, VG, k_blocks, kb128;
    int w_stages, x_stages;
    int dual;  // two MMA issuers, two accumulators (bf16, one 128-token tile)
    uint32_t w_stage_bytes, x_stage_bytes, x_bytes;
    int gather;  // gather the hash rows in this launch
    const int32_t* ids;
    int64_t ids_stride;
    const int64_t* row_offset;
    const int64_t* rows;
    const uint16_t* table;   // bf16 rows, or e4m3 codes of an fp8 table
    const uint8_t* tscale;   // fp8 table: ue8m0 [rows][E/32]; else null
    uint16_t* staged;       // [rows_alloc][K] bf16
    uint8_t* staged_q;      // MXFP8: e4m3 codes [rows_alloc][K]
    uint8_t* staged_s;      // MXFP8: scale atoms of the codes
    const uint8_t* wscale;  // MXFP8: E8M0 [N/32][K/32]
    const uint16_t* hidden;
    int64_t hs_t, hs_h;
    uint16_t* out;
    int64_t os_t, os_h;
    const uint8_t* mask;
    const float* qk;       // [H, D]
    const uint8_t* wpack;  // [K bytes/128][N][128 bytes], CTA slices consecutive
    float4* rec;           // records (shh, skk, shk, -) per copy block [Tpitch][nh]
    int rec_base[kMaxCopies];  // float4 offset of each copy's block
    int cf[kMaxCopies];        // first CTA holding each copy's keys
    int nh[kMaxCopies];        // number of CTAs holding each copy's keys
    float* value;              // fp32 [T][D]: each CTA's value dims, read by the residual items
    uint16_t* kv;              // kv mode: bf16 [T][kv_ld] keys then value; no gate, no residual
    int64_t kv_ld;
    unsigned long long* bar;   // launch counter, then three barrier counters
    float* gate_out;
    float eps, clamp, inv_d, inv_sqrt_d;
    unsigned* err;
    uint32_t x_off, qk_off, bar_off;
    int hv8;  // hidden rows and strides 32-byte aligned: 32-byte loads
};

__device__ __forceinline__ int first_granule(int cta, int n, int G) {
    return static_cast<int>(static_cast<int64_t>(cta) * n / G);
}

// 16 fp32 values (bit patterns) -> 16 bf16 (nearest even) at dst, 32-byte
// aligned: two 16-byte stores.
__device__ __forceinline__ void store_bf16x16(uint16_t* dst, const uint32_t (&r)[16]) {
    uint4 o[2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
        o[h] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * h + 0]), __uint_as_float(r[8 * h + 1])),
                          pack_bf16x2(__uint_as_float(r[8 * h + 2]), __uint_as_float(r[8 * h + 3])),
                          pack_bf16x2(__uint_as_float(r[8 * h + 4]), __uint_as_float(r[8 * h + 5])),
                          pack_bf16x2(__uint_as_float(r[8 * h + 6]), __uint_as_float(r[8 * h + 7])));
    st_v4(dst, o[0]);
    st_v4(dst + 8, o[1]);
}

__device__ __forceinline__ void fail(int* abort_flag, unsigned* err) {
    *reinterpret_cast<volatile int*>(abort_flag) = 1;
    atomicOr(err, ENGRAM_DEVERR_TIMEOUT);
}

// Grid barrier: a posted release add, then a bounded wait until all G CTAs
// of this launch (epoch e) have arrived.  One thread per CTA.
__device__ __forceinline__ void grid_arrive(unsigned long long* ctr) {
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(ctr) : "memory");
}

__device__ __forceinline__ bool grid_wait(const unsigned long long* ctr, unsigned long long target) {
    const uint64_t t0 = globaltimer_ns();
    uint32_t spins = 0;
    while (ld_acquire_u64(ctr) < target) {
        __nanosleep(32);
        if ((++spins & 15u) == 0 &&
            (globaltimer_ns() - t0 > kWaitLimitNs || spins > kWaitLimitIters))
            return false;
    }
    return true;
}

template <bool kMx, bool kF8T>
__global__ void __launch_bounds__(kThreads, 1)
    decode_fused_kernel(const __grid_constant__ CUtensorMap tm_x, const FusedArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* xring = smem + a.x_off;
    float* qk_s = reinterpret_cast<float*>(smem + a.qk_off);  // q*k of the slice's key columns
    uint64_t* wfull = reinterpret_cast<uint64_t*>(smem + a.bar_off);
    uint64_t* wempty = wfull + kMaxWStages;
    uint64_t* xfull = wempty + kMaxWStages;
    uint64_t* xempty = xfull + kMaxXStages;
    uint64_t* tfull = xempty + kMaxXStages;  // every MMA done
    uint64_t* drain = tfull + 1;
    uint64_t* drain2 = drain + 1;  // the second issuer's in-flight MMAs
    uint64_t* scbar = drain2 + 1;         // MXFP8: every scale word is in TMEM
    unsigned long long* epoch_s = reinterpret_cast<unsigned long long*>(scbar + 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epoch_s + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
    const volatile int* abort_v = abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int G = gridDim.x;
    const int c = blockIdx.x;
    // this CTA's columns: value dims [v0, v0 + vlen), key columns [k0, k0 + klen)
    const int g0 = first_granule(c, a.NG, G), g1 = first_granule(c + 1, a.NG, G);
    const int vg0 = first_granule(c, a.VG, G), vg1 = first_granule(c + 1, a.VG, G);
    const int v0 = vg0 * 16, vlen = (vg1 - vg0) * 16;
    const int k0 = (g0 - vg0) * 16, klen = ((g1 - vg1) - (g0 - vg0)) * 16;
    const int width = vlen + klen;  // a multiple of 16, at most kMaxFusedSlice
    const int c_lo = g0 * 16;       // first packed row
    const uint32_t w_bytes = static_cast<uint32_t>(width) * 128u;

    // Gather item i of this CTA (a 16-byte chunk of a hash row; MXFP8: a
    // 32-k block, four chunks): the id, then the row.  Each gathering
    // thread fetches its first two items before the CTA-wide setup below, so
    // the dependent id -> row loads overlap it and each other.
    const int nrows_g = a.T * a.C;
    const int g_r0 = static_cast<int>(static_cast<int64_t>(c) * nrows_g / G);
    const int g_r1 = static_cast<int>(static_cast<int64_t>(c + 1) * nrows_g / G);
    const int g_per = kMx ? (a.E >> 5) : (a.E >> 3);  // items per hash row
    const int g_n = a.gather ? (g_r1 - g_r0) * g_per : 0;
    auto fetch = [&](int i, uint4 (&v)[4]) -> bool {
        const int rr = g_r0 + i / g_per, b = i - (i / g_per) * g_per;
        const int t = rr / a.C, cc = rr - t * a.C;
        const int64_t id = a.ids[t * a.ids_stride + cc];
        const bool good = id >= 0 && id < __ldg(a.rows + cc);
        const int64_t row = __ldg(a.row_offset + cc) + (good ? id : 0);
        if constexpr (kF8T) {  // fp8 table: dequantize on the way
            const uint8_t* cp = reinterpret_cast<const uint8_t*>(a.table) + row * a.E + b * (kMx ? 32 : 8);
            const uint32_t sb = good ? __ldg(a.tscale + row * (a.E >> 5) + (kMx ? b : (b >> 2))) : 0u;
#pragma unroll
            for (int j = 0; j < (kMx ? 4 : 1); ++j)
                v[j] = good ? dequant8(__ldg(reinterpret_cast<const uint2*>(cp + j * 8)), sb)
                            : make_uint4(0u, 0u, 0u, 0u);
            return good;
        }
        const uint16_t* src = a.table + row * a.E + b * (kMx ? 32 : 8);
#pragma unroll
        for (int j = 0; j < (kMx ? 4 : 1); ++j)
            v[j] = good ? ld_stream_v4(src + j * 8) : make_uint4(0u, 0u, 0u, 0u);
        return good;
    };
    if (tid == 0) {
        for (int s = 0; s < a.w_stages; ++s) {
            mbar_init(&wfull[s], 1);
            mbar_init(&wempty[s], 1);
        }
        for (int s = 0; s < a.x_stages; ++s) {
            mbar_init(&xfull[s], 1);  // the loading thread's expect_tx
            mbar_init(&xempty[s], 1);
        }
        mbar_init(tfull, a.dual ? 2 : 1);  // one commit per issuer
        mbar_init(drain, 1);
        mbar_init(drain2, 1);
        mbar_init(scbar, 128);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tm_x);
        pdl_launch_dependents();
    }
    int w_issued = 0;
    int x_issued = 0;  // token-tile copies issued (thread 64)
    const uint64_t pol_w = policy_evict_first();
    const uint8_t* w_src = a.wpack + static_cast<int64_t>(c_lo) * 128;
    const int64_t w_kstep = static_cast<int64_t>(a.N) * 128;
    if (tid == 0) {
        // the first ring of weight stages needs no free slot: issue it now
        for (; w_issued < a.w_stages && w_issued < a.k_blocks; ++w_issued) {
            mbar_arrive_expect_tx(&wfull[w_issued], w_bytes);
            bulk_load_hint(smem + w_issued * a.w_stage_bytes, w_src, w_bytes, &wfull[w_issued],
                           pol_w);
            w_src += w_kstep;
        }
    }
    // everything below may read what the preceding launch wrote
    pdl_wait();
    if (tid == 0) {
        // this launch's epoch: stable until CTA 0 advances it at the end
        *epoch_s = *reinterpret_cast<volatile unsigned long long*>(a.bar) + 1ull;
    }
    // (a thread's second item too, so that two id -> row chains overlap when
    // rows cross the host link)
    uint4 pre[4] = {}, pre2[4] = {};
    bool pre_good = true, pre2_good = true;
    if (warp >= 2 && warp < 6 && tid - 64 < g_n) pre_good = fetch(tid - 64, pre);
    if constexpr (!kMx)  // (MXFP8: one item per thread ahead; a second one measured slower;
                         // the gather loop below fetches any further items either way)
        if (warp >= 2 && warp < 6 && tid - 64 + 128 < g_n) pre2_good = fetch(tid - 64 + 128, pre2);
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const unsigned long long target = *epoch_s * static_cast<unsigned long long>(G);
    // MXFP8 scale cells, 8 columns per k-block each (every region 8-aligned)
    const uint32_t tm_sfa = tmem_base + kMaxFusedSlice;                     // tokens
    const uint32_t tm_sfb = tm_sfa + 8u * static_cast<uint32_t>(a.kb128);  // weights

    const bool kvm = a.kv != nullptr;  // kv mode: hidden, mask and out are not read
    // This CTA's residual items after grid barrier 2: (token, 256-dim block)
    // pairs [i0, i1) of the T * D/256 in token-major order.
    const int nb = a.D >> 8;
    const int n_items = kvm ? 0 : a.T * nb;
    const int it0 = static_cast<int>(static_cast<int64_t>(c) * n_items / G);
    const int it1 = static_cast<int>(static_cast<int64_t>(c + 1) * n_items / G);

    if (warp == 0) {
        if (lane == 0) {
            // the rest of the weight slice, a stage as soon as its MMAs are done
            bool ok = true;
            int s = 0;
            uint32_t par = 1;  // the second use of each stage
            for (int kb = w_issued; kb < a.k_blocks; ++kb) {
                if (!mbar_wait_sleep(&wempty[s], par ^ 1u, abort_v, 128)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&wfull[s], w_bytes);
                bulk_load_hint(smem + s * a.w_stage_bytes, w_src, w_bytes, &wfull[s], pol_w);
                w_src += w_kstep;
                ++w_issued;
                if (++s == a.w_stages) {
                    s = 0;
                    par ^= 1u;
                }
            }
            if (!ok) fail(abort_flag, a.err);
        }
    } else if (warp == 1 || (warp == 6 && a.dual)) {
        if (lane == 0) {
            // An issuing thread's dependent scalar work
            // sets the pace: stage indices, phase parities and shared-memory
            // descriptors advance incrementally (a descriptor's address field
            // is the byte address / 16), and each k-block's MMAs are unrolled.
            const uint32_t idesc = idesc_bf16(128, width);
            uint32_t idm[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) idm[k] = idesc_mxf8(128, width, k, k);
            const uint64_t wdesc0 = smem_desc_sw128(smem_addr(smem));
            const uint64_t xdesc0 = smem_desc_sw128(smem_addr(xring));
            const uint64_t wstep = a.w_stage_bytes >> 4, xstep = a.x_stage_bytes >> 4;
            const bool two_tiles = a.mtiles == 2;
            bool ok = true;
            if constexpr (kMx) {
                ok = mbar_wait(scbar, 0, abort_v);
                tc_fence_after();
            }
            // this issuer's k-blocks and accumulator
            const int kstep = a.dual ? 2 : 1;
            const int kb0 = warp == 6 ? 1 : 0;
            const uint32_t dacc = tmem_base + (warp == 6 ? 256u : 0u);
            int sw = 0, sx = 0;
            uint32_t pw = 0, px = 0, acc = 0;
            uint64_t wd = wdesc0, xd = xdesc0;
            uint32_t sfa = tm_sfa, sfb = tm_sfb;
            auto advance = [&]() {
                if (++sw == a.w_stages) {
                    sw = 0;
                    pw ^= 1u;
                    wd = wdesc0;
                } else {
                    wd += wstep;
                }
                if (++sx == a.x_stages) {
                    sx = 0;
                    px ^= 1u;
                    xd = xdesc0;
                } else {
                    xd += xstep;
                }
            };
            if (kb0 == 1) advance();
            for (int kb = kb0; kb < a.k_blocks && ok; kb += kstep) {
                if (!mbar_wait(&wfull[sw], pw, abort_v) || !mbar_wait(&xfull[sx], px, abort_v)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if constexpr (kMx) {
                    // 4 x K32, scale byte k of each cell
                    mma_mxf8_ss(tmem_base, xd, wd, idm[0], sfa, sfb, acc);
                    mma_mxf8_ss(tmem_base, xd + 2, wd + 2, idm[1], sfa, sfb, 1u);
                    mma_mxf8_ss(tmem_base, xd + 4, wd + 4, idm[2], sfa, sfb, 1u);
                    mma_mxf8_ss(tmem_base, xd + 6, wd + 6, idm[3], sfa, sfb, 1u);
                    sfa += 8u;
                    sfb += 8u;
                } else {
                    // 4 x K16; the second 128-token tile 16 KB on
                    mma_bf16_ss(dacc, xd, wd, idesc, acc);
                    if (two_tiles) mma_bf16_ss(tmem_base + kMaxFusedSlice, xd + 1024, wd, idesc, acc);
#pragma unroll
                    for (int k = 1; k < 4; ++k) {
                        mma_bf16_ss(dacc, xd + 2 * k, wd + 2 * k, idesc, 1u);
                        if (two_tiles)
                            mma_bf16_ss(tmem_base + kMaxFusedSlice, xd + 1024 + 2 * k, wd + 2 * k,
                                        idesc, 1u);
                    }
                }
                acc = 1u;
                mma_commit(&wempty[sw]);
                mma_commit(&xempty[sx]);
                advance();
                if (kstep == 2) advance();  // skip the other issuer's k-block
            }
            if (ok) mma_commit(tfull);
            if (!ok) fail(abort_flag, a.err);
        }
    } else if (warp < 6) {
        const int etid = tid - 64;  // 0..127 (warps 2-5; warp 6 idles unless it issues MMAs)
        const int q = warp & 3;     // TMEM lane quarter of this warp
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        if constexpr (kMx) {
            // weight scales of the slice: B row j (slice column j) in lane
            // j % 32, column tm_sfb + 8 kb + j / 32; every lane quarter gets
            // a copy
            for (int kb = 0; kb < a.kb128; ++kb) {
                uint32_t w[8];
#pragma unroll
                for (int jc = 0; jc < 8; ++jc) {
                    const int j = jc * 32 + lane;
                    const int n = j < vlen ? a.H * a.D + v0 + j : k0 + (j - vlen);
                    w[jc] = j < width ? __ldg(reinterpret_cast<const uint32_t*>(
                                            a.wscale + (n >> 5) * (a.K >> 5) + kb * 4))
                                      : 0x7F7F7F7Fu;
                }
                const uint32_t col = tm_sfb + lane_base + 8u * static_cast<uint32_t>(kb);
                tmem_st4(col, w[0], w[1], w[2], w[3]);
                tmem_st4(col + 4, w[4], w[5], w[6], w[7]);
            }
        }
        // q*k of the slice's key columns (fixed at create)
        for (int j = etid; j < klen; j += 128) qk_s[j] = __ldg(a.qk + k0 + j);
        // This CTA's share of the hash rows -> the staged-rows buffer
        // (ParallelEngramEmbedding.lookup); MXFP8: also their e4m3 codes and
        // scales.  Every CTA's token tiles need every row: grid barrier 1.
        if (a.gather) {
            bool bad = false;
            for (int i = etid; i < g_n; i += 128) {
                uint4 v[4];
                bool good;
                if (i == etid) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) v[j] = pre[j];
                    good = pre_good;
                } else if (!kMx && i == etid + 128) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) v[j] = pre2[j];
                    good = pre2_good;
                } else {
                    good = fetch(i, v);
                }
                bad |= !good;
                const int rr = g_r0 + i / g_per, b = i - (i / g_per) * g_per;
                if constexpr (kMx) {
                    const int t = rr / a.C, cc = rr - t * a.C;
                    const int64_t k0r = static_cast<int64_t>(rr) * a.E + b * 32;  // t*K + c*E + 32b
#pragma unroll
                    for (int j = 0; j < 4; ++j) st_v4(a.staged + k0r + j * 8, v[j]);
                    uint4 cq[2];
                    const uint32_t sb = mx_quantize32(v, cq);
                    st_v4(a.staged_q + k0r, cq[0]);
                    st_v4(a.staged_q + k0r + 16, cq[1]);
                    a.staged_s[sf_atom_offset(t, (cc * a.E + b * 32) >> 5, a.kb128)] =
                        static_cast<uint8_t>(sb);
                } else {
                    st_v4(a.staged + static_cast<int64_t>(rr) * a.E + b * 8, v[0]);
                }
            }
            if (bad) atomicOr(a.err, ENGRAM_DEVERR_BAD_HASH_ID);
            fence_proxy_async();  // other CTAs read these rows with TMA copies
        }
        // grid barrier 1 (the counter advances on every launch, gather or not)
        named_barrier_sync(1, 128);
        if (etid == 0) {
            grid_arrive(a.bar + 1);
            if (a.gather && !grid_wait(a.bar + 1, target)) fail(abort_flag, a.err);
        }
        named_barrier_sync(1, 128);  // qk_s complete; grid barrier 1 has passed
        // Token tiles: k-block kb of the first Tn staged rows into stage
        // kb % x_stages by one TMA box (128-row boxes for a second tile), row
        // r at 128 * r, 16-byte chunk j at position j ^ (r % 8): the 128-byte
        // swizzle the MMA descriptors expect.  Rows past T hold whatever is
        // staged there; their accumulator rows are never used.  (MXFP8: the
        // token scales go to TMEM once the first tiles are on their way.)
        {
            // MXFP8 token scales: A row r = token t in lane t, column
            // tm_sfa + 8 kb + t / 32 (written to all four columns); needed
            // before the first MMA, written once the first tiles are in flight
            constexpr int kMaxKb128 = 16;  // (TMEM budget: 256 + 16 * K/128 <= 512)
            uint32_t sfw[kMaxKb128];
            auto token_scales = [&]() {
#pragma unroll
                for (int b = 0; b < kMaxKb128; ++b)
                    if (b < a.kb128)
                        tmem_st4(tm_sfa + lane_base + 8u * static_cast<uint32_t>(b), sfw[b],
                                 sfw[b], sfw[b], sfw[b]);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(scbar);
            };
            constexpr int kKElems = kMx ? 128 : 64;  // elements per 128-byte row of a k-block
            bool ok = true;
            auto load_x = [&](int kb) {  // thread 64 only
                const int s = kb % a.x_stages;
                uint8_t* xs = xring + s * a.x_stage_bytes;
                mbar_arrive_expect_tx(&xfull[s], a.x_bytes);
                tma_load_2d(xs, &tm_x, &xfull[s], kb * kKElems, 0);
                if (a.mtiles == 2) tma_load_2d(xs + 16384, &tm_x, &xfull[s], kb * kKElems, 128);
                ++x_issued;
            };
            const int first = a.k_blocks < a.x_stages ? a.k_blocks : a.x_stages;
            if (etid == 0) {
                fence_proxy_async();  // the staged rows were written by ordinary stores
                for (int kb = 0; kb < first; ++kb) load_x(kb);
            }
            __syncwarp();
            // (after the first tiles: the proxy fence would wait for these loads)
            if constexpr (kMx) {
                const int t = q * 32 + lane;
#pragma unroll
                for (int b = 0; b < kMaxKb128; ++b)
                    sfw[b] = b < a.kb128 ? __ldcg(reinterpret_cast<const unsigned*>(
                                               a.staged_s + sf_atom_offset(t, 4 * b, a.kb128)))
                                         : 0u;
            }
            if (kMx) token_scales();  // (the first MMAs wait for the scales)
            if (etid == 0) {
                // the rest, each as soon as its stage's MMAs are done
                for (int kb = first; kb < a.k_blocks; ++kb) {
                    const int s = kb % a.x_stages;
                    if (!mbar_wait_sleep(&xempty[s],
                                         static_cast<uint32_t>((kb / a.x_stages) & 1) ^ 1u, abort_v,
                                         64)) {
                        ok = false;
                        break;
                    }
                    load_x(kb);
                }
                if (!ok) fail(abort_flag, a.err);
            }
            __syncwarp();
        }

        // Epilogue: thread = one token of an accumulator, key columns of the
        // slice -> one record per (hc copy, token).
        const int h0 = k0 / a.D;  // the key run covers copies h0 and possibly h0 + 1
        bool go = true;
        for (int m = 0; m < a.mtiles && go; ++m) {
            const int t = m * 128 + q * 32 + lane;
            const bool live = t < a.T;
            // this token's hidden at the key columns, before the accumulator is ready
            uint4 hv[2 * kKeyChunks];
#pragma unroll
            for (int ci = 0; ci < kKeyChunks; ++ci) {
                hv[2 * ci] = hv[2 * ci + 1] = make_uint4(0u, 0u, 0u, 0u);
                if (live && !kvm && ci * 16 < klen) {
                    const int n0 = k0 + ci * 16;
                    const int h = n0 / a.D, d0 = n0 - h * a.D;
                    const uint16_t* hp = a.hidden + t * a.hs_t + h * a.hs_h + d0;
                    if (a.hv8) {
                        ld_nc_v8(hp, hv[2 * ci], hv[2 * ci + 1]);
                    } else {
                        hv[2 * ci] = ld_nc_v4(hp);
                        hv[2 * ci + 1] = ld_nc_v4(hp + 8);
                    }
                }
            }
            if (m == 0) {
                const bool bad = !mbar_wait_sleep(tfull, 0, abort_v, 128);
                // all four epilogue warps decide together
                if (named_barrier_or(1, 128, bad || *abort_v)) {
                    if (bad) fail(abort_flag, a.err);
                    go = false;
                    break;
                }
                tc_fence_after();
            }
            float acc[2][3] = {{0.f, 0.f, 0.f}, {0.f, 0.f, 0.f}};
            const uint32_t taddr =
                tmem_base + lane_base + static_cast<uint32_t>(m * kMaxFusedSlice + vlen);
#pragma unroll
            for (int ci = 0; ci < kKeyChunks; ++ci) {
                if (ci * 16 >= klen) break;
                uint32_t r[16];
                tmem_ld16(taddr + static_cast<uint32_t>(ci * 16), r);
                if (a.dual) {
                    uint32_t r2[16];
                    tmem_ld16(taddr + 256u + static_cast<uint32_t>(ci * 16), r2);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(r2[e]));
                }
                tmem_ld_wait();
                if (kvm) {
                    if (live) store_bf16x16(a.kv + static_cast<int64_t>(t) * a.kv_ld + k0 + ci * 16, r);
                    continue;
                }
                const int n0 = k0 + ci * 16;  // 16 columns never straddle an hc copy
                const int hi = n0 / a.D - h0;
                const uint32_t w[8] = {hv[2 * ci].x,     hv[2 * ci].y,     hv[2 * ci].z,
                                       hv[2 * ci].w,     hv[2 * ci + 1].x, hv[2 * ci + 1].y,
                                       hv[2 * ci + 1].z, hv[2 * ci + 1].w};
                float shh = 0.f, skk = 0.f, shk = 0.f;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float x = (e & 1) ? bf16hi(w[e >> 1]) : bf16lo(w[e >> 1]);
                    const float key = __uint_as_float(r[e]);
                    shh = fmaf(x, x, shh);
                    skk = fmaf(key, key, skk);
                    shk = fmaf(x * qk_s[ci * 16 + e], key, shk);
                }
                acc[hi][0] += shh;
                acc[hi][1] += skk;
                acc[hi][2] += shk;
            }
            if (live && !kvm) {
                // a record for every copy whose CTA range includes this CTA
                // (zeros where it holds none of the copy's keys)
                const int hl = klen > 0 ? (k0 + klen - 1) / a.D : -1;  // last copy of the run
                for (int h = 0; h < a.H; ++h) {
                    if (c < a.cf[h] || c >= a.cf[h] + a.nh[h]) continue;
                    const bool has = h >= h0 && h <= hl;
                    a.rec[a.rec_base[h] + t * a.nh[h] + (c - a.cf[h])] =
                        has ? make_float4(acc[h - h0][0], acc[h - h0][1], acc[h - h0][2], 0.f)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            if (kvm) {
                for (int ci = 0; ci * 16 < vlen; ++ci) {
                    uint32_t r[16];  // every lane loads (tcgen05.ld is warp-wide)
                    const uint32_t va =
                        tmem_base + lane_base + static_cast<uint32_t>(m * kMaxFusedSlice + ci * 16);
                    tmem_ld16(va, r);
                    if (a.dual) {
                        uint32_t r2[16];
                        tmem_ld16(va + 256u, r2);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(r2[e]));
                    }
                    tmem_ld_wait();
                    if (live)
                        store_bf16x16(a.kv + static_cast<int64_t>(t) * a.kv_ld +
                                          static_cast<int64_t>(a.H) * a.D + v0 + ci * 16,
                                      r);
                }
            }
            if (!kvm) {
                // the fp32 value of this CTA's dims for every token: the residual
                // items after grid barrier 2 read it from L2
                for (int ci = 0; ci * 16 < vlen; ++ci) {
                    uint32_t r[16];
                    const uint32_t va =
                        tmem_base + lane_base + static_cast<uint32_t>(m * kMaxFusedSlice + ci * 16);
                    tmem_ld16(va, r);
                    if (a.dual) {
                        uint32_t r2[16];
                        tmem_ld16(va + 256u, r2);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(r2[e]));
                    }
                    tmem_ld_wait();
                    if (live) {
                        float4* vp = reinterpret_cast<float4*>(
                            a.value + static_cast<int64_t>(t) * a.D + v0 + ci * 16);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            vp[e] = make_float4(__uint_as_float(r[4 * e]),
                                                __uint_as_float(r[4 * e + 1]),
                                                __uint_as_float(r[4 * e + 2]),
                                                __uint_as_float(r[4 * e + 3]));
                    }
                }
            }
        }
        // the residual items' hidden rows towards L2 (read after barrier 2;
        // plain per-line prefetches, four 128-byte lines per copy and item)
        if (go)
            for (int l = etid; l < (it1 - it0) * a.H * 4; l += 128) {
                const int item = it0 + l / (a.H * 4), r = l - (l / (a.H * 4)) * (a.H * 4);
                const int t = item / nb, d = (item - t * nb) * 256 + (r & 3) * 64;
                prefetch_line_l2(a.hidden + t * a.hs_t + (r >> 2) * a.hs_h + d);
            }
        // every record this CTA owes is written: grid barrier 2 (the release
        // add of one thread covers the CTA's writes ordered before it by the
        // named barrier)
        named_barrier_sync(1, 128);
        if (etid == 0) {
            grid_arrive(a.bar + 2);
            if (!grid_wait(a.bar + 2, target)) fail(abort_flag, a.err);
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    // Residual items: every CTA finishes its (token, 256-dim block) items
    // straight after grid barrier 2.  Each thread first loads its task (8
    // dims of one item: the fp32 value and the H hidden chunks); warps reduce
    // the gate of every (token, copy) its items touch from the records (lane
    // l adds records l, l + 32, ..., then a shuffle tree: a fixed order, so
    // runs are bit-identical) into shared memory; then out = hidden +
    // gate * value (masked tokens keep hidden's bits).  The records, the
    // value and hidden all come in one round trip, and no CTA waits for
    // another's gates.
    float* gate_s = qk_s;  // (the q*k slice is no longer needed)
    const int tok0 = it1 > it0 ? it0 / nb : 0;
    const int ntok = it1 > it0 ? (it1 - 1) / nb - tok0 + 1 : 0;
    if (!*abort_v && ntok > 0) {
        const int ntask = (it1 - it0) * 32;
        auto task_at = [&](int k, int& t, int& d) {
            const int item = it0 + (k >> 5);
            t = item / nb;
            d = (item - t * nb) * 256 + (k & 31) * 8;
        };
        // the first task's operands, before the gates
        float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
        uint4 x[kMaxCopies];
        int t0 = 0, d0 = 0;
        const bool has0 = tid < ntask;
        if (has0) {
            task_at(tid, t0, d0);
            const float4* vp = reinterpret_cast<const float4*>(a.value + static_cast<int64_t>(t0) * a.D + d0);
            v0 = __ldcg(vp);
            v1 = __ldcg(vp + 1);
#pragma unroll
            for (int h = 0; h < kMaxCopies; ++h)
                if (h < a.H) x[h] = ld_nc_v4(a.hidden + t0 * a.hs_t + h * a.hs_h + d0);
        }
        // (two rows per warp at a time, their records loaded together, so a
        // CTA whose items touch two tokens still takes one round trip)
        for (int r0 = warp; r0 < ntok * a.H; r0 += 2 * kWarps) {
            float acc[2][3] = {{0.f, 0.f, 0.f}, {0.f, 0.f, 0.f}};
            const int nrow = r0 + kWarps < ntok * a.H ? 2 : 1;
            const float4* rr[2];
            int nhr[2], tr[2], hr_[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int r = r0 + k * kWarps;
                tr[k] = tok0 + (k < nrow ? r / a.H : 0);
                hr_[k] = k < nrow ? r - (r / a.H) * a.H : 0;
                nhr[k] = k < nrow ? a.nh[hr_[k]] : 0;
                rr[k] = a.rec + a.rec_base[hr_[k]] + static_cast<int64_t>(tr[k]) * nhr[k];
            }
            const int nmax = nhr[0] > nhr[1] ? nhr[0] : nhr[1];
            for (int j = lane; j < nmax; j += 32) {
                float4 v[2];
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    v[k] = j < nhr[k] ? __ldcg(rr[k] + j) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    if (j >= nhr[k]) continue;
                    acc[k][0] += v[k].x;
                    acc[k][1] += v[k].y;
                    acc[k][2] += v[k].z;
                }
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                float s_hh = acc[k][0], s_kk = acc[k][1], s_hk = acc[k][2];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    s_hh += __shfl_xor_sync(0xFFFFFFFFu, s_hh, o);
                    s_kk += __shfl_xor_sync(0xFFFFFFFFu, s_kk, o);
                    s_hk += __shfl_xor_sync(0xFFFFFFFFu, s_hk, o);
                }
                if (lane == 0 && k < nrow) {
                    const int t = tr[k], h = hr_[k];
                    const bool active = a.mask == nullptr || a.mask[t] != 0;
                    const float hr = 1.0f / sqrtf(s_hh * a.inv_d + a.eps);
                    const float kr = 1.0f / sqrtf(s_kk * a.inv_d + a.eps);
                    const float dot = s_hk * hr * kr * a.inv_sqrt_d;
                    float gi = sqrtf(fmaxf(fabsf(dot), a.clamp));
                    if (dot < 0.0f) gi = -gi;
                    const float g = active ? 1.0f / (1.0f + expf(-gi)) : 0.0f;
                    gate_s[r0 + k * kWarps] = g;
                    a.gate_out[t * a.H + h] = g;  // (CTAs sharing a token write the same bits)
                }
            }
        }
        __syncthreads();
        auto finish = [&](int t, int d, const float4& va, const float4& vb, const uint4 (&xh)[kMaxCopies]) {
            const bool active = a.mask == nullptr || a.mask[t] != 0;
            const float v[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
#pragma unroll
            for (int h = 0; h < kMaxCopies; ++h) {
                if (h >= a.H) continue;
                uint4 o = xh[h];
                if (active) {
                    const float g = gate_s[(t - tok0) * a.H + h];
                    const uint32_t w[4] = {o.x, o.y, o.z, o.w};
                    uint32_t p[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        p[k] = pack_bf16x2(fmaf(g, v[2 * k], bf16lo(w[k])),
                                           fmaf(g, v[2 * k + 1], bf16hi(w[k])));
                    o = make_uint4(p[0], p[1], p[2], p[3]);
                }
                st_v4(a.out + t * a.os_t + h * a.os_h + d, o);
            }
        };
        if (has0) finish(t0, d0, v0, v1, x);
        for (int k = tid + kThreads; k < ntask; k += kThreads) {
            int t, d;
            task_at(k, t, d);
            const float4* vp = reinterpret_cast<const float4*>(a.value + static_cast<int64_t>(t) * a.D + d);
            const float4 va = __ldcg(vp), vb = __ldcg(vp + 1);
            uint4 xh[kMaxCopies];
#pragma unroll
            for (int h = 0; h < kMaxCopies; ++h)
                if (h < a.H) xh[h] = ld_nc_v4(a.hidden + t * a.hs_t + h * a.hs_h + d);
            finish(t, d, va, vb, xh);
        }
    }
    if (*abort_v) {
        // let in-flight copies and MMAs land before shared memory and TMEM go
        if (tid == 0) {
            for (int j = w_issued > a.w_stages ? w_issued - a.w_stages : 0; j < w_issued; ++j)
                mbar_wait(&wfull[j % a.w_stages], static_cast<uint32_t>((j / a.w_stages) & 1),
                          nullptr);
        }
        if (tid == 64) {
            for (int j = x_issued > a.x_stages ? x_issued - a.x_stages : 0; j < x_issued; ++j)
                mbar_wait(&xfull[j % a.x_stages], static_cast<uint32_t>((j / a.x_stages) & 1),
                          nullptr);
        }
        if (tid == 32) {
            mma_commit(drain);
            mbar_wait(drain, 0, nullptr);
        }
        if (tid == 192 && a.dual) {
            mma_commit(drain2);
            mbar_wait(drain2, 0, nullptr);
        }
        __syncthreads();
        tc_fence_after();
        if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
        return;
    }
    tc_fence_after();

    // every CTA read this launch's epoch before its barrier 2 arrival, and
    // this CTA passed barrier 2: advance it
    if (c == 0 && tid == 0) atomicAdd(a.bar, 1ull);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// wkv [N, row_bytes] -> [row_bytes/128][N][128 bytes] in the fused kernel's
// column order (each CTA's value rows, then its key rows, CTA after CTA):
// for every 128-byte k-block (64 bf16 or 128 e4m3) the rows are consecutive
// 128-byte lines, each 8-row group 128-byte swizzled (16-byte chunk j of
// packed row p at position j ^ (p % 8)), so a CTA's rows of a k-block are a
// ready shared-memory operand image.
__global__ void pack_w_kernel(const uint8_t* w, uint8_t* wp, int64_t N, int64_t row_bytes, int D,
                              int H, int NG, int VG, int G) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // 16-B chunk
    const int64_t cpr = row_bytes / 16;
    if (i >= N * cpr) return;
    const int64_t p = i / cpr;  // packed row
    const int64_t ch = i - p * cpr;
    const int x = static_cast<int>(p >> 4);                                        // granule
    const int cta = static_cast<int>((static_cast<int64_t>(x + 1) * G - 1) / NG);  // its owner
    const int g0 = first_granule(cta, NG, G), vg0 = first_granule(cta, VG, G);
    const int vlen = (first_granule(cta + 1, VG, G) - vg0) * 16;
    const int j = static_cast<int>(p - static_cast<int64_t>(g0) * 16);  // slice column
    const int64_t n = j < vlen ? static_cast<int64_t>(H) * D + vg0 * 16 + j
                               : static_cast<int64_t>(g0 - vg0) * 16 + (j - vlen);
    const int64_t kb = ch / 8, jj = ch % 8;
    const int64_t dst = (kb * N + p) * 128 + ((jj ^ (p & 7)) * 16);
    *reinterpret_cast<uint4*>(wp + dst) = *reinterpret_cast<const uint4*>(w + n * row_bytes + ch * 16);
}

int host_first(int cta, int n, int G) { return static_cast<int>(static_cast<int64_t>(cta) * n / G); }

}  // namespace

FusedLayout fused_layout(int64_t N, int64_t D, int64_t H, int num_sms) {
    FusedLayout L = {};
    L.NG = static_cast<int>(N / 16);
    L.VG = static_cast<int>(D / 16);
    L.grid = num_sms < L.NG ? num_sms : L.NG;
    L.ok = H >= 1 && H <= kMaxCopies && L.grid >= 1;
    int last_cta[kMaxCopies];
    for (int h = 0; h < kMaxCopies; ++h) {
        L.cf[h] = L.nh[h] = 0;
        last_cta[h] = -1;
    }
    for (int c = 0; c < L.grid && L.ok; ++c) {
        const int g0 = host_first(c, L.NG, L.grid), g1 = host_first(c + 1, L.NG, L.grid);
        const int vg0 = host_first(c, L.VG, L.grid), vg1 = host_first(c + 1, L.VG, L.grid);
        const int kg0 = g0 - vg0, kg1 = g1 - vg1;
        const int width = (g1 - g0) * 16;
        if (kg1 < kg0 || width > kMaxFusedSlice) {
            L.ok = false;
            break;
        }
        if (width > L.max_width) L.max_width = width;
        if (kg1 > kg0) {
            const int hf = static_cast<int>(kg0 * 16 / D);
            const int hl = static_cast<int>((kg1 * 16 - 1) / D);
            if (hl - hf > 1) L.ok = false;  // a key run spans at most two copies
            for (int h = hf; h <= hl && h < kMaxCopies; ++h) {
                if (last_cta[h] < 0) L.cf[h] = c;
                last_cta[h] = c;
            }
        }
    }
    for (int h = 0; h < H && L.ok; ++h) {
        if (last_cta[h] < 0)
            L.ok = false;
        else
            L.nh[h] = last_cta[h] - L.cf[h] + 1;
    }
    return L;
}

// Shared memory of one launch: weight ring | token ring | q*k slice |
// barriers, from the 1024-byte aligned base.
FusedSmem fused_smem(const FusedLayout& L, const FusedPlan& p, bool mx) {
    FusedSmem m = {};
    if (!L.ok || L.max_width <= 0 || p.mtiles < 1) return m;  // no launch: ok stays false
    m.x_bytes = static_cast<uint32_t>(p.mtiles == 1 ? p.Tn * 128 : 2 * 16384);
    m.x_stage_bytes = (m.x_bytes + 1023u) / 1024u * 1024u;
    m.w_stage_bytes = static_cast<uint32_t>((L.max_width * 128 + 1023) / 1024 * 1024);
    const uint32_t qk_bytes = kMaxFusedSlice * 4, bar_bytes = 1024;
    const uint32_t budget = kFusedSmemBytes - 1024;  // after 1024-byte alignment
    // The MMA reads all 128 rows of a token tile (M = 128) even when T is
    // smaller; rows past T are never used, but the last stage's 16 KB read
    // must stay inside this CTA's shared memory.
    // Token stages: about kXRingTarget bytes of them (at least 4), so that
    // the tiles in flight cover the L2 round trip of the refills.
    int xs = static_cast<int>(kXRingTarget / m.x_stage_bytes);
    xs = xs < 4 ? 4 : (xs > kMaxXStages ? kMaxXStages : xs);
    m.x_stages = xs;
    m.x_ring = static_cast<uint32_t>(xs) * m.x_stage_bytes;
    if (p.mtiles == 1 && m.x_ring < static_cast<uint32_t>(xs - 1) * m.x_stage_bytes + 16384u)
        m.x_ring = static_cast<uint32_t>(xs - 1) * m.x_stage_bytes + 16384u;
    const uint32_t fixed = m.x_ring + qk_bytes + bar_bytes;
    int stages = fixed < budget ? static_cast<int>((budget - fixed) / m.w_stage_bytes) : 0;
    if (stages > kMaxWStages) stages = kMaxWStages;
    m.ok = stages >= 2;
    m.w_stages = stages;
    m.dual = (!mx && p.mtiles == 1) ? 1 : 0;
    m.x_off = static_cast<uint32_t>(stages) * m.w_stage_bytes;
    m.qk_off = m.x_off + m.x_ring;
    m.bar_off = m.qk_off + qk_bytes;
    // after barrier 2 the q*k area holds the gates of the tokens a CTA's
    // residual items touch
    const int nb = L.VG * 16 / 256, items = (p.Tn * nb + L.grid - 1) / L.grid;
    if ((items / (nb > 0 ? nb : 1) + 2) * kMaxCopies > kMaxFusedSlice) m.ok = false;
    return m;
}

FusedPlan fused_plan(const engram_handle* h, int64_t T) {
    FusedPlan p = {};
    p.Tn = static_cast<int>((T + 15) / 16 * 16);
    p.mtiles = static_cast<int>((T + 127) / 128);
    p.k_blocks = static_cast<int>(h->K * (h->cfg.wkv_format == ENGRAM_WKV_MXFP8 ? 1 : 2) / 128);
    return p;
}

bool fused_supported(const engram_handle* h, int64_t T) {
    if (!h->fused.ok) return false;
    if (h->cfg.wkv_format == ENGRAM_WKV_MXFP8) {
        // one accumulator of 256 columns plus 8 + 8 scale columns per k-block
        return T >= 1 && T <= kMaxFusedTMx && h->cfg.head_dim % 32 == 0 &&
               kMaxFusedSlice + 16 * (h->K / 128) <= 512;
    }
    return T >= 1 && T <= kMaxFusedT && h->cfg.head_dim % 8 == 0;
}

cudaError_t pack_weights(const engram_handle* h, cudaStream_t s) {
    if (!h->fused.ok) return cudaSuccess;  // the fused kernel will not run
    const int64_t row_bytes = h->K * (h->cfg.wkv_format == ENGRAM_WKV_MXFP8 ? 1 : 2);
    const int64_t nchunks = h->N * row_bytes / 16;
    pack_w_kernel<<<static_cast<unsigned>((nchunks + 255) / 256), 256, 0, s>>>(
        static_cast<const uint8_t*>(h->wkv), h->ws.wpack, h->N, row_bytes,
        static_cast<int>(h->cfg.dim), static_cast<int>(h->cfg.hc_mult), h->fused.NG, h->fused.VG,
        h->fused.grid);
    return cudaGetLastError();
}

cudaError_t fused_setup_attributes() {
    const void* fns[] = {reinterpret_cast<const void*>(decode_fused_kernel<false, false>),
                         reinterpret_cast<const void*>(decode_fused_kernel<false, true>),
                         reinterpret_cast<const void*>(decode_fused_kernel<true, false>),
                         reinterpret_cast<const void*>(decode_fused_kernel<true, true>)};
    for (const void* fn : fns) {
        const cudaError_t e =
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmemBytes);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_fused_debug_value(const engram_handle* h, float* value, int64_t T,
                                     cudaStream_t s) {
    return cudaMemcpyAsync(value, h->ws.fvalue, T * h->cfg.dim * sizeof(float),
                           cudaMemcpyDeviceToDevice, s);
}

cudaError_t launch_decode_fused(engram_handle* h, const void* hidden, const int64_t* hs,
                                const int32_t* ids, int64_t ids_stride, const uint8_t* mask,
                                void* out, const int64_t* os, int64_t T, cudaStream_t s,
                                bool pdl, uint16_t* kv, int64_t kv_ld) {
    const FusedPlan p = fused_plan(h, T);
    const FusedLayout& L = h->fused;
    const bool mx = h->cfg.wkv_format == ENGRAM_WKV_MXFP8;
    const bool f8t = h->table_scale != nullptr;
    FusedArgs a = {};
    a.T = static_cast<int>(T);
    a.Tn = p.Tn;
    a.D = static_cast<int>(h->cfg.dim);
    a.H = static_cast<int>(h->cfg.hc_mult);
    a.C = static_cast<int>(h->C);
    a.E = static_cast<int>(h->cfg.head_dim);
    a.N = static_cast<int>(h->N);
    a.K = static_cast<int>(h->K);
    a.mtiles = p.mtiles;
    a.NG = L.NG;
    a.VG = L.VG;
    a.k_blocks = p.k_blocks;
    a.kb128 = static_cast<int>(h->K / 128);
    a.gather = ids != nullptr ? 1 : 0;
    a.ids = ids;
    a.ids_stride = ids_stride;
    a.row_offset = h->d_row_offset;
    a.rows = h->d_rows;
    a.table = h->table;
    a.tscale = h->table_scale;
    a.staged = h->ws.staged;
    a.staged_q = h->ws.staged_q;
    a.staged_s = h->ws.staged_s;
    a.wscale = h->wkv_scale;
    a.hidden = static_cast<const uint16_t*>(hidden);
    a.hs_t = hs != nullptr ? hs[0] : 0;
    a.hs_h = hs != nullptr ? hs[1] : 0;
    // (key runs start on 16-dim granules, so aligned rows keep 32-byte loads aligned)
    a.hv8 = (reinterpret_cast<uintptr_t>(hidden) % 32 == 0 && a.hs_t % 16 == 0 &&
             a.hs_h % 16 == 0) ? 1 : 0;
    a.out = static_cast<uint16_t*>(out);
    a.os_t = os != nullptr ? os[0] : 0;
    a.os_h = os != nullptr ? os[1] : 0;
    a.mask = mask;
    a.kv = kv;  // kv mode: hidden, out and mask unused
    a.kv_ld = kv_ld;
    a.qk = h->ws.qk;
    a.wpack = h->ws.wpack;
    a.rec = reinterpret_cast<float4*>(h->ws.fpart);
    int base = 0;
    for (int hh = 0; hh < kMaxCopies; ++hh) {
        a.cf[hh] = L.cf[hh];
        a.nh[hh] = L.nh[hh];
        a.rec_base[hh] = base;
        base += static_cast<int>(h->ws.kv_tpitch) * L.nh[hh];
    }
    a.value = h->ws.fvalue;  // the value exchange buffer of the residual items
    a.bar = reinterpret_cast<unsigned long long*>(h->ws.grid_bar);
    a.gate_out = h->ws.gate;
    a.eps = static_cast<float>(h->cfg.eps);
    a.clamp = static_cast<float>(h->cfg.clamp);
    a.inv_d = 1.0f / static_cast<float>(a.D);
    a.inv_sqrt_d = 1.0f / sqrtf(static_cast<float>(a.D));
    a.err = h->ws.err;
    const FusedSmem m = fused_smem(L, p, mx);
    if (!m.ok) return cudaErrorInvalidConfiguration;
    a.x_bytes = m.x_bytes;
    a.x_stage_bytes = m.x_stage_bytes;
    a.w_stage_bytes = m.w_stage_bytes;
    a.x_stages = m.x_stages;
    a.w_stages = m.w_stages;
    a.dual = m.dual;
    a.x_off = m.x_off;
    a.qk_off = m.qk_off;
    a.bar_off = m.bar_off;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(L.grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kFusedSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    // token tiles: a box of Tn rows, or two of 128
    CUtensorMap tm_x = p.mtiles == 1 ? h->tm_act_n[p.Tn / 16 - 1] : h->tm_act_m;
    void* args[] = {&tm_x, &a};
    return cudaLaunchKernelExC(
        &cfg,
        mx ? (f8t ? reinterpret_cast<const void*>(decode_fused_kernel<true, true>)
                  : reinterpret_cast<const void*>(decode_fused_kernel<true, false>))
           : (f8t ? reinterpret_cast<const void*>(decode_fused_kernel<false, true>)
                  : reinterpret_cast<const void*>(decode_fused_kernel<false, false>)),
        args);
}

}  // namespace engram
