// The whole Engram forward of a decode step (T <= 256) in one cooperative,
// persistent kernel (one CTA per SM).  Engram.forward
// ("vllm.models.deepseek_v4_1.common.engram") defines the layer; the gate
// arithmetic is that of _engram_gate_finish_kernel with one rank
// ("vllm.models.deepseek_v41.amd.engram").
//
// Work split: CTA i owns a contiguous slice of the projection's N = D*(H+1)
// columns -- 16-column granules dealt out evenly, so 128 or 144 columns at
// the decode shapes -- over the full K.  Tokens sit on the MMA's M side
// (128 rows per accumulator; rows past T are ignored), the slice on N.
//
//   gather   every CTA copies its share (about 1/grid) of the T x C hash
//            rows into the staged-rows buffer (an id outside its table
//            gives a zero row and sets the device error flag), so each SM
//            touches only a few of the table's pages; then a first grid
//            barrier.  The weight stream has started meanwhile.  Rows
//            staged by an earlier engram_lookup skip this step;
//   wkv      wkv is packed at create time k-block-major with the 128-byte
//            swizzle applied, so each stage's weight slice is one contiguous
//            bulk copy; the staged token rows arrive by TMA (a box of T
//            rows rounded up to 16); tcgen05 kind::f16, fp32 accumulators in
//            TMEM;
//   epilogue each thread owns one token's whole slice (its hidden columns
//            are loaded while the MMAs run): for key columns it sums
//            hidden^2, key^2 and hidden*q*k*key per hc copy (the split over
//            dim that _engram_gate_partials_kernel uses across ranks, here
//            across CTAs), for value columns it stores the value;
//   finish   after a second grid barrier each CTA takes (token, hc) rows:
//            one warp per row adds the partial sums of the CTAs covering
//            that hc copy (a fixed order: results are run-to-run identical)
//            and forms the signed-sqrt sigmoid gate; then all threads write
//            hidden + gate * value (masked tokens copy hidden's bits).  The
//            value rows and partial records arrive by bulk copy; the hidden
//            rows were bulk-copied while the weights streamed.
//
// MXFP8 wkv (T <= 128): the gather also quantises the rows (e4m3 codes and
// E8M0 scales per 32 k), the MMAs are tcgen05 kind::mxf8f6f4 with
// block_scale, and the scale factors sit in TMEM next to the accumulator.
// A CTA's weight slice starts on any 16-column boundary, so instead of
// copying scale atoms the epilogue warps write the scale words into TMEM
// themselves (tcgen05.st): the weights' at kernel start, the tokens' after
// the gather.  Scale cell layout (tcgen05 block scaling, scale_vec::1X):
// the scale of A row r for k-block b sits in lane r, column sfa + r / 32,
// byte b; that of B row n in lane n % 32, column sfb + n / 32, byte b.
//
// Both grid barriers reset themselves, so a captured launch replays.
#include <cuda_bf16.h>

#include "internal.h"
#include "mxfp8.cuh"
#include "ptx.cuh"

namespace engram {
namespace {

constexpr int kThreads = 192;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxStages = 8;
constexpr int kSliceChunks = kMaxFusedSlice / 16;  // 16-column chunks of one slice
constexpr int kPartFloats = 8;  // per (token, CTA): 2 hc copies x (hh, kk, hk, pad)
constexpr int kHidRows = 4;     // finish rows whose hidden is prefetched to shared memory

struct FusedArgs {
    int T, Tn, D, H, C, E, N, K;
    int mtiles, granules, k_blocks, stages;
    int kb128;  // K / 128: MXFP8 scale words per row
    uint32_t w_stage_bytes, x_bytes;  // per stage: weight slice region, token bytes
    int gather;                       // gather the hash rows in this launch
    const int32_t* ids;
    int64_t ids_stride;
    const int64_t* row_offset;
    const int64_t* rows;
    const uint16_t* table;
    uint16_t* staged;    // [rows_alloc][K] bf16
    uint8_t* staged_q;   // MXFP8: e4m3 codes [rows_alloc][K]
    uint8_t* staged_s;   // MXFP8: scale atoms of the codes
    const uint8_t* wscale;  // MXFP8: E8M0 [N/32][K/32]
    const uint16_t* hidden;
    int64_t hs_t, hs_h;
    uint16_t* out;
    int64_t os_t, os_h;
    const uint8_t* mask;
    const float* qk;        // [H, D]
    const uint8_t* wpack;   // [K bytes/128][N][128 bytes], 8-row groups 128-byte swizzled
    float* part;            // [tpitch][grid][kPartFloats]
    float* value;           // [tpitch][D]
    unsigned* bar;          // two grid barriers: {arrivals, generation} each
    float* gate_out;
    float eps, clamp, inv_d, inv_sqrt_d;
    unsigned* err;
    uint32_t hid_off, qk_off, bar_off, hid_rows;
};

// CTA that owns granule x when NG granules are dealt to G CTAs.
__device__ __forceinline__ int owner(int x, int NG, int G) { return ((x + 1) * G - 1) / NG; }
__device__ __forceinline__ int first_granule(int cta, int NG, int G) {
    return static_cast<int>(static_cast<int64_t>(cta) * NG / G);
}

__device__ __forceinline__ void fail(int* abort_flag, unsigned* err) {
    *reinterpret_cast<volatile int*>(abort_flag) = 1;
    atomicOr(err, ENGRAM_DEVERR_TIMEOUT);
}

// Self-resetting grid barrier: the last CTA to arrive zeroes the count and
// advances the generation; the others wait, bounded, for the generation
// to change.  One thread per CTA, after the CTA's writes are fenced.
__device__ __forceinline__ bool grid_barrier(unsigned* bar, unsigned G) {
    const unsigned gen = ld_acquire_u32(bar + 1);
    __threadfence();
    if (atomicAdd(bar, 1u) == G - 1u) {
        bar[0] = 0u;
        __threadfence();
        atomicAdd(bar + 1, 1u);
        return true;
    }
    const uint64_t t0 = globaltimer_ns();
    uint32_t spins = 0;
    while (ld_acquire_u32(bar + 1) == gen) {
        if ((++spins & 63u) == 0 &&
            (globaltimer_ns() - t0 > kWaitLimitNs || spins > kWaitLimitIters))
            return false;
    }
    return true;
}

template <bool kMx>
__global__ void __launch_bounds__(kThreads, 1)
    decode_fused_kernel(const __grid_constant__ CUtensorMap tm_x, const FusedArgs a) {
    constexpr int kKElems = kMx ? 128 : 64;  // k per 128-byte block
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t stage_bytes = a.w_stage_bytes + a.mtiles * 16384u;
    uint16_t* hid_s = reinterpret_cast<uint16_t*>(smem + a.hid_off);
    float* qk_s = reinterpret_cast<float*>(smem + a.qk_off);  // the slice's q*k columns
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.bar_off);
    uint64_t* empty = full + kMaxStages;
    uint64_t* tfull = empty + kMaxStages;
    uint64_t* hbar = tfull + 1;
    uint64_t* fbar = hbar + 1;
    uint64_t* drain = fbar + 1;
    uint64_t* scbar = drain + 1;  // MXFP8: every scale word is in TMEM
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(scbar + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
    float* gate_s = reinterpret_cast<float*>(abort_flag + 2);  // [kWarps] gates of a row batch
    const volatile int* abort_v = abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int G = gridDim.x;
    const int HR = a.T * a.H;  // (token, hc) rows of the output
    const int c_lo = first_granule(blockIdx.x, a.granules, G) * 16;  // this CTA's slice
    const int c_hi = first_granule(blockIdx.x + 1, a.granules, G) * 16;
    const int width = c_hi - c_lo;  // a multiple of 16, at most kMaxFusedSlice
    const uint32_t w_bytes = static_cast<uint32_t>(width) * 128u;

    if (tid == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(hbar, 1);
        mbar_init(fbar, 1);
        mbar_init(drain, 1);
        mbar_init(scbar, 128);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tm_x);
    }
    // generation of the gather barrier, read before this CTA can arrive at it
    const unsigned gather_gen = (a.gather && tid == 0) ? ld_acquire_u32(a.bar + 1) : 0u;
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // MXFP8 scale cells, 8 columns per k-block each (every region 8-aligned)
    const uint32_t tm_sfa = tmem_base + kMaxFusedSlice;                     // tokens
    const uint32_t tm_sfb = tm_sfa + 8u * static_cast<uint32_t>(a.kb128);  // weights

    int issued = 0;
    if (warp == 0) {
        if (lane == 0) {
            // hidden rows of this CTA's share of the finish, while weights stream
            int nh = 0;
            for (int r = blockIdx.x; r < HR && nh < static_cast<int>(a.hid_rows); r += G) ++nh;
            if (nh > 0) {
                mbar_arrive_expect_tx(hbar, static_cast<uint32_t>(nh * a.D * 2));
                int i = 0;
                for (int r = blockIdx.x; r < HR && i < nh; r += G, ++i) {
                    const int t = r / a.H, h = r - t * a.H;
                    bulk_load(hid_s + static_cast<int64_t>(i) * a.D,
                              a.hidden + t * a.hs_t + h * a.hs_h, static_cast<uint32_t>(a.D * 2),
                              hbar);
                }
            } else {
                mbar_arrive(hbar);
            }
            const uint64_t pol_w = policy_evict_first();
            // token tiles wait for the staged rows (the first grid barrier);
            // the weight slices of the first stages go out at once
            bool have_rows = !a.gather;
            auto issue_x = [&](int s, int kb) {
                uint8_t* sx = smem + s * stage_bytes + a.w_stage_bytes;
                for (int m = 0; m < a.mtiles; ++m)
                    tma_load_2d(sx + m * 16384, &tm_x, &full[s], kb * kKElems, m * 128);
            };
            auto await_rows = [&]() -> bool {
                const uint64_t t0 = globaltimer_ns();
                uint32_t spins = 0;
                while (ld_acquire_u32(a.bar + 1) == gather_gen) {
                    if ((++spins & 63u) == 0 &&
                        (*abort_v || globaltimer_ns() - t0 > kWaitLimitNs || spins > kWaitLimitIters))
                        return false;
                }
                fence_proxy_async();  // the staged rows were written by ordinary stores
                for (int j = 0; j < issued; ++j) issue_x(j % a.stages, j);
                have_rows = true;
                return true;
            };
            bool ok = true;
            for (int kb = 0; kb < a.k_blocks && ok; ++kb) {
                if (!have_rows && issued == a.stages && !await_rows()) {
                    ok = false;
                    break;
                }
                const int s = issued % a.stages;
                const uint32_t par = static_cast<uint32_t>((issued / a.stages) & 1);
                if (!mbar_wait(&empty[s], par ^ 1u, abort_v)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], w_bytes + a.x_bytes);
                bulk_load_hint(smem + s * stage_bytes,
                               a.wpack + (static_cast<int64_t>(kb) * a.N + c_lo) * 128, w_bytes,
                               &full[s], pol_w);
                if (have_rows) issue_x(s, kb);
                ++issued;
            }
            if (ok && !have_rows && !await_rows()) ok = false;
            if (!ok) fail(abort_flag, a.err);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(128, width);
            bool ok = true;
            if constexpr (kMx) {
                ok = mbar_wait(scbar, 0, abort_v);
                tc_fence_after();
            }
            for (int kb = 0; kb < a.k_blocks && ok; ++kb) {
                const int s = kb % a.stages;
                if (!mbar_wait(&full[s], static_cast<uint32_t>((kb / a.stages) & 1), abort_v)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sw = smem_addr(smem + s * stage_bytes);
                const uint64_t wdesc = smem_desc_sw128(sw);
                if constexpr (kMx) {
                    const uint64_t xdesc = smem_desc_sw128(sw + a.w_stage_bytes);
#pragma unroll
                    for (int k = 0; k < 4; ++k)  // 4 x K32, scale byte k of each cell
                        mma_mxf8_ss(tmem_base, xdesc + 2 * k, wdesc + 2 * k,
                                    idesc_mxf8(128, width, k, k),
                                    tm_sfa + 8u * static_cast<uint32_t>(kb),
                                    tm_sfb + 8u * static_cast<uint32_t>(kb),
                                    (kb > 0 || k > 0) ? 1u : 0u);
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        for (int m = 0; m < a.mtiles; ++m)
                            mma_bf16_ss(tmem_base + static_cast<uint32_t>(m * kMaxFusedSlice),
                                        smem_desc_sw128(sw + a.w_stage_bytes + m * 16384) + 2 * k,
                                        wdesc + 2 * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(&empty[s]);
            }
            if (ok) mma_commit(tfull);
            if (!ok) fail(abort_flag, a.err);
        }
    } else {
        const int etid = tid - 64;  // 0..127
        const int q = warp & 3;     // TMEM lane quarter of this warp
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        if constexpr (kMx) {
            // weight scales of the slice: B row n (slice column n) in lane
            // n % 32, column tm_sfb + 8 kb + n / 32; every lane quarter gets
            // a copy
            for (int kb = 0; kb < a.kb128; ++kb) {
                uint32_t w[8];
#pragma unroll
                for (int jc = 0; jc < 8; ++jc) {
                    const int n = jc * 32 + lane;
                    w[jc] = n < width ? __ldg(reinterpret_cast<const uint32_t*>(
                                            a.wscale + ((c_lo + n) >> 5) * (a.K >> 5) + kb * 4))
                                      : 0x7F7F7F7Fu;
                }
                const uint32_t col = tm_sfb + lane_base + 8u * static_cast<uint32_t>(kb);
                tmem_st4(col, w[0], w[1], w[2], w[3]);
                tmem_st4(col + 4, w[4], w[5], w[6], w[7]);
            }
        }
        // This CTA's share of the hash rows -> the staged-rows buffer
        // (ParallelEngramEmbedding.lookup), then the first grid barrier.
        if (a.gather && kMx) {
            // one thread per 32-k block of a hash row: the bf16 row, its
            // e4m3 codes and its scale
            const int bpr = a.E >> 5;
            const int nrows = a.T * a.C;
            const int r0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * nrows / G);
            const int r1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * nrows / G);
            bool bad = false;
            for (int i = etid; i < (r1 - r0) * bpr; i += 128) {
                const int rr = r0 + i / bpr, b = i - (i / bpr) * bpr;
                const int t = rr / a.C, c = rr - t * a.C;
                const int64_t id = a.ids[t * a.ids_stride + c];
                uint4 v[4];
                if (id >= 0 && id < __ldg(a.rows + c)) {
                    const uint16_t* src = a.table + (__ldg(a.row_offset + c) + id) * a.E + b * 32;
#pragma unroll
                    for (int j = 0; j < 4; ++j) v[j] = ld_stream_v4(src + j * 8);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) v[j] = make_uint4(0u, 0u, 0u, 0u);
                    bad = true;
                }
                const int64_t k0 = static_cast<int64_t>(rr) * a.E + b * 32;  // = t*K + c*E + 32b
#pragma unroll
                for (int j = 0; j < 4; ++j) st_v4(a.staged + k0 + j * 8, v[j]);
                uint4 cq[2];
                const uint32_t sb = mx_quantize32(v, cq);
                st_v4(a.staged_q + k0, cq[0]);
                st_v4(a.staged_q + k0 + 16, cq[1]);
                a.staged_s[sf_atom_offset(t, (c * a.E + b * 32) >> 5, a.kb128)] =
                    static_cast<uint8_t>(sb);
            }
            if (bad) atomicOr(a.err, ENGRAM_DEVERR_BAD_HASH_ID);
            __threadfence();
            named_barrier_sync(1, 128);
            if (etid == 0 && !grid_barrier(a.bar, static_cast<unsigned>(G))) fail(abort_flag, a.err);
        } else if (a.gather) {
            const int cpr = a.E >> 3;  // 16-byte chunks per row
            const int nrows = a.T * a.C;
            const int r0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * nrows / G);
            const int r1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * nrows / G);
            bool bad = false;
            for (int q = etid; q < (r1 - r0) * cpr; q += 128) {
                const int rr = r0 + q / cpr, j = q - (q / cpr) * cpr;
                const int t = rr / a.C, c = rr - t * a.C;
                const int64_t id = a.ids[t * a.ids_stride + c];
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (id >= 0 && id < __ldg(a.rows + c))
                    v = ld_stream_v4(a.table + (__ldg(a.row_offset + c) + id) * a.E + j * 8);
                else
                    bad = true;
                st_v4(a.staged + static_cast<int64_t>(rr) * a.E + j * 8, v);
            }
            if (bad) atomicOr(a.err, ENGRAM_DEVERR_BAD_HASH_ID);
            __threadfence();
            named_barrier_sync(1, 128);
            if (etid == 0 && !grid_barrier(a.bar, static_cast<unsigned>(G))) fail(abort_flag, a.err);
        }
        // q*k of the slice's key columns (q*k is [H][D], i.e. columns [0, H*D))
        for (int c = etid; c < width; c += 128) {
            const int n = c_lo + c;
            qk_s[c] = n < a.H * a.D ? __ldg(a.qk + n) : 0.f;
        }
        named_barrier_sync(1, 128);  // qk_s complete; the gather barrier has passed
        if constexpr (kMx) {
            // token scales: A row r = token t in lane t, column
            // tm_sfa + 8 kb + t / 32 (written to all four columns)
            const int t = q * 32 + lane;
            for (int kb = 0; kb < a.kb128; ++kb) {
                const uint32_t w = __ldcg(reinterpret_cast<const unsigned*>(
                    a.staged_s + sf_atom_offset(t, 4 * kb, a.kb128)));
                tmem_st4(tm_sfa + lane_base + 8u * static_cast<uint32_t>(kb), w, w, w, w);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(scbar);
        }

        // Epilogue: thread = one token of an accumulator (TMEM lane quarter
        // = warp % 4), columns = the slice.
        const int h0 = c_lo / a.D;  // the slice covers hc copies h0 and possibly h0 + 1
        bool go = true;
        for (int m = 0; m < a.mtiles && go; ++m) {
            const int t = m * 128 + q * 32 + lane;
            const bool live = t < a.T;
            // this token's hidden columns of the slice, before the accumulator is ready
            uint4 hv[2 * kSliceChunks];
#pragma unroll
            for (int ci = 0; ci < kSliceChunks; ++ci) {
                const int n0 = c_lo + ci * 16;
                hv[2 * ci] = hv[2 * ci + 1] = make_uint4(0u, 0u, 0u, 0u);
                if (live && ci * 16 < width && n0 < a.H * a.D) {
                    const int h = n0 / a.D, d0 = n0 - h * a.D;
                    const uint16_t* hp = a.hidden + t * a.hs_t + h * a.hs_h + d0;
                    hv[2 * ci] = ld_nc_v4(hp);
                    hv[2 * ci + 1] = ld_nc_v4(hp + 8);
                }
            }
            if (m == 0) {
                const bool bad = !mbar_wait(tfull, 0, abort_v);
                // all four epilogue warps decide together
                if (named_barrier_or(1, 128, bad || *abort_v)) {
                    if (bad) fail(abort_flag, a.err);
                    go = false;
                    break;
                }
                tc_fence_after();
            }
            float acc[2][3] = {{0.f, 0.f, 0.f}, {0.f, 0.f, 0.f}};
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(m * kMaxFusedSlice);
#pragma unroll
            for (int ci = 0; ci < kSliceChunks; ++ci) {
                if (ci * 16 >= width) break;
                uint32_t r[16];
                tmem_ld16(taddr + static_cast<uint32_t>(ci * 16), r);
                tmem_ld_wait();
                if (!live) continue;
                const int n0 = c_lo + ci * 16;  // 16 columns never straddle an hc copy
                const int h = n0 / a.D, d0 = n0 - h * a.D;
                if (h < a.H) {
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
                    const int hi = h - h0;
                    acc[hi][0] += shh;
                    acc[hi][1] += skk;
                    acc[hi][2] += shk;
                } else {
                    float4* vp =
                        reinterpret_cast<float4*>(a.value + static_cast<int64_t>(t) * a.D + d0);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        vp[e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                                            __uint_as_float(r[4 * e + 2]),
                                            __uint_as_float(r[4 * e + 3]));
                }
            }
            if (live) {
                float4* pp = reinterpret_cast<float4*>(
                    a.part + (static_cast<int64_t>(t) * G + blockIdx.x) * kPartFloats);
                pp[0] = make_float4(acc[0][0], acc[0][1], acc[0][2], 0.f);
                pp[1] = make_float4(acc[1][0], acc[1][1], acc[1][2], 0.f);
            }
        }
        // every partial sum and value this CTA owes is written
        __threadfence();
        named_barrier_sync(1, 128);
        if (etid == 0 && !grid_barrier(a.bar + 2, static_cast<unsigned>(G))) fail(abort_flag, a.err);
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (*abort_v) {
        // let in-flight copies and MMAs land before shared memory and TMEM go
        if (tid == 0) {
            const int first = issued > a.stages ? issued - a.stages : 0;
            for (int j = first; j < issued; ++j)
                mbar_wait(&full[j % a.stages], static_cast<uint32_t>((j / a.stages) & 1), nullptr);
        }
        if (tid == 32) {
            mma_commit(drain);
            mbar_wait(drain, 0, nullptr);
        }
    }
    // the hidden rows were bulk-copied at the start; they must have landed
    if (!mbar_wait(hbar, 0, nullptr) && lane == 0) fail(abort_flag, a.err);
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
    if (*abort_v) return;

    // Finish.  Rows of this CTA: r = blockIdx.x + i * G.  Lane i of warp 0
    // copies row i's value row and the partial records of the CTAs covering
    // its hc copy into the (idle) stage buffers.
    const int nchunk = a.D >> 3;
    float* fin = reinterpret_cast<float*>(smem);  // per row: [D value][G records]
    const int64_t per_row = a.D + static_cast<int64_t>(G) * kPartFloats;
    int nrows = 0;
    for (int r = blockIdx.x; r < HR; r += G) ++nrows;
    if (warp == 0 && nrows > 0) {
        uint32_t bytes = 0;
        int t = 0, h = 0, cf = 0, cl = 0;
        const bool mine = lane < nrows;
        if (mine) {
            const int r = blockIdx.x + lane * G;
            t = r / a.H;
            h = r - t * a.H;
            cf = owner(h * a.D / 16, a.granules, G);
            cl = owner(((h + 1) * a.D - 1) / 16, a.granules, G);
            bytes = static_cast<uint32_t>(a.D * 4 + (cl - cf + 1) * kPartFloats * 4);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) bytes += __shfl_xor_sync(0xFFFFFFFFu, bytes, off);
        if (lane == 0) mbar_arrive_expect_tx(fbar, bytes);
        __syncwarp();
        if (mine) {
            fence_proxy_async();  // written by other CTAs, read by bulk copies
            float* dst = fin + static_cast<int64_t>(lane) * per_row;
            bulk_load(dst, a.value + static_cast<int64_t>(t) * a.D, static_cast<uint32_t>(a.D * 4),
                      fbar);
            bulk_load(dst + a.D + cf * kPartFloats,
                      a.part + (static_cast<int64_t>(t) * G + cf) * kPartFloats,
                      static_cast<uint32_t>((cl - cf + 1) * kPartFloats * 4), fbar);
        }
    }
    if (nrows > 0 && !mbar_wait(fbar, 0, nullptr)) {
        if (lane == 0) fail(abort_flag, a.err);
    }
    for (int b0 = 0; b0 < nrows; b0 += kWarps) {
        // one warp per row: the partial sums of the CTAs covering hc copy h,
        // lane l taking CTAs cf + l, cf + l + 32, ..., then a shuffle tree
        const int i = b0 + warp;
        if (i < nrows) {
            const int r = blockIdx.x + i * G;
            const int t = r / a.H, h = r - t * a.H;
            const float* recs = fin + static_cast<int64_t>(i) * per_row + a.D;
            const int cf = owner(h * a.D / 16, a.granules, G);
            const int cl = owner(((h + 1) * a.D - 1) / 16, a.granules, G);
            float s_hh = 0.f, s_kk = 0.f, s_hk = 0.f;
            for (int cta = cf + lane; cta <= cl; cta += 32) {
                const int hfirst = first_granule(cta, a.granules, G) * 16 / a.D;
                const float* p = recs + cta * kPartFloats + (h == hfirst ? 0 : 4);
                s_hh += p[0];
                s_kk += p[1];
                s_hk += p[2];
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                s_hh += __shfl_xor_sync(0xFFFFFFFFu, s_hh, off);
                s_kk += __shfl_xor_sync(0xFFFFFFFFu, s_kk, off);
                s_hk += __shfl_xor_sync(0xFFFFFFFFu, s_hk, off);
            }
            if (lane == 0) {
                const bool active = a.mask == nullptr || a.mask[t] != 0;
                const float hr = 1.0f / sqrtf(s_hh * a.inv_d + a.eps);
                const float kr = 1.0f / sqrtf(s_kk * a.inv_d + a.eps);
                const float dot = s_hk * hr * kr * a.inv_sqrt_d;
                float gi = sqrtf(fmaxf(fabsf(dot), a.clamp));
                if (dot < 0.0f) gi = -gi;
                const float g = active ? 1.0f / (1.0f + expf(-gi)) : 0.0f;
                gate_s[warp] = g;
                a.gate_out[r] = g;
            }
        }
        __syncthreads();
        const int nb = nrows - b0 < kWarps ? nrows - b0 : kWarps;
        for (int w = 0; w < nb; ++w) {
            const int i2 = b0 + w;
            const int r = blockIdx.x + i2 * G;
            const int t = r / a.H, h = r - t * a.H;
            const bool active = a.mask == nullptr || a.mask[t] != 0;
            const float g = gate_s[w];
            const uint16_t* hrow = i2 < static_cast<int>(a.hid_rows)
                                       ? hid_s + static_cast<int64_t>(i2) * a.D
                                       : a.hidden + t * a.hs_t + h * a.hs_h;
            const float* vrow = fin + static_cast<int64_t>(i2) * per_row;
            uint16_t* orow = a.out + t * a.os_t + h * a.os_h;
            for (int c = tid; c < nchunk; c += kThreads) {
                const int d = c * 8;
                uint4 o = *reinterpret_cast<const uint4*>(hrow + d);
                if (active) {
                    const float4 v0 = *reinterpret_cast<const float4*>(vrow + d);
                    const float4 v1 = *reinterpret_cast<const float4*>(vrow + d + 4);
                    const uint32_t w4[4] = {o.x, o.y, o.z, o.w};
                    o.x = pack_bf16x2(fmaf(g, v0.x, bf16lo(w4[0])), fmaf(g, v0.y, bf16hi(w4[0])));
                    o.y = pack_bf16x2(fmaf(g, v0.z, bf16lo(w4[1])), fmaf(g, v0.w, bf16hi(w4[1])));
                    o.z = pack_bf16x2(fmaf(g, v1.x, bf16lo(w4[2])), fmaf(g, v1.y, bf16hi(w4[2])));
                    o.w = pack_bf16x2(fmaf(g, v1.z, bf16lo(w4[3])), fmaf(g, v1.w, bf16hi(w4[3])));
                }
                st_v4(orow + d, o);
            }
        }
        __syncthreads();  // gate_s is reused by the next batch
    }
}

// wkv [N, row_bytes] -> [row_bytes/128][N][128 bytes]: for every 128-byte
// k-block (64 bf16 or 128 e4m3) the rows are consecutive 128-byte lines,
// each 8-row group 128-byte swizzled (16-byte chunk j of row n at position
// j ^ (n % 8)), so any 8-aligned row range of a k-block is a ready
// shared-memory operand image.
__global__ void pack_w_kernel(const uint8_t* w, uint8_t* wp, int64_t N, int64_t row_bytes) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // 16-B chunk
    const int64_t cpr = row_bytes / 16;
    if (i >= N * cpr) return;
    const int64_t n = i / cpr;
    const int64_t c = i - n * cpr;
    const int64_t kb = c / 8, j = c % 8;
    const int64_t dst = (kb * N + n) * 128 + ((j ^ (n & 7)) * 16);
    *reinterpret_cast<uint4*>(wp + dst) = *reinterpret_cast<const uint4*>(w + i * 16);
}

}  // namespace

FusedPlan fused_plan(const engram_handle* h, int64_t T) {
    FusedPlan p = {};
    p.Tn = static_cast<int>((T + 15) / 16 * 16);
    p.mtiles = static_cast<int>((T + 127) / 128);
    p.granules = static_cast<int>(h->N / 16);
    p.k_blocks = static_cast<int>(h->K * (h->cfg.wkv_format == ENGRAM_WKV_MXFP8 ? 1 : 2) / 128);
    p.grid = h->num_sms < p.granules ? h->num_sms : p.granules;
    p.max_width = (p.granules + p.grid - 1) / p.grid * 16;  // widest slice
    return p;
}

bool fused_supported(const engram_handle* h, int64_t T) {
    const FusedPlan p = fused_plan(h, T);
    if (h->cfg.wkv_format == ENGRAM_WKV_MXFP8) {
        // one accumulator of 256 columns plus 8 + 8 scale columns per k-block
        return T >= 1 && T <= kMaxFusedTMx && p.max_width <= kMaxFusedSlice &&
               h->cfg.head_dim % 32 == 0 && kMaxFusedSlice + 16 * (h->K / 128) <= 512;
    }
    return T >= 1 && T <= kMaxFusedT && p.max_width <= kMaxFusedSlice && h->cfg.head_dim % 8 == 0;
}

cudaError_t pack_weights(const engram_handle* h, cudaStream_t s) {
    const int64_t row_bytes = h->K * (h->cfg.wkv_format == ENGRAM_WKV_MXFP8 ? 1 : 2);
    const int64_t nchunks = h->N * row_bytes / 16;
    pack_w_kernel<<<static_cast<unsigned>((nchunks + 255) / 256), 256, 0, s>>>(
        static_cast<const uint8_t*>(h->wkv), h->ws.wpack, h->N, row_bytes);
    return cudaGetLastError();
}

cudaError_t fused_setup_attributes() {
    cudaError_t e = cudaFuncSetAttribute(decode_fused_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kFusedSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(decode_fused_kernel<true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmemBytes);
}

cudaError_t launch_fused_debug_value(const engram_handle* h, float* value, int64_t T,
                                     cudaStream_t s) {
    return cudaMemcpyAsync(value, h->ws.fvalue, T * h->cfg.dim * sizeof(float),
                           cudaMemcpyDeviceToDevice, s);
}

cudaError_t launch_decode_fused(engram_handle* h, const void* hidden, const int64_t* hs,
                                const int32_t* ids, int64_t ids_stride, const uint8_t* mask,
                                void* out, const int64_t* os, int64_t T, cudaStream_t s) {
    const FusedPlan p = fused_plan(h, T);
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
    a.granules = p.granules;
    a.k_blocks = p.k_blocks;
    a.kb128 = static_cast<int>(h->K / 128);
    // token rows per stage: one box of Tn rows, or two of 128 rows
    a.x_bytes = static_cast<uint32_t>(p.mtiles == 1 ? p.Tn * 128 : 2 * 16384);
    a.gather = ids != nullptr ? 1 : 0;
    a.ids = ids;
    a.ids_stride = ids_stride;
    a.row_offset = h->d_row_offset;
    a.rows = h->d_rows;
    a.table = h->table;
    a.staged = h->ws.staged;
    a.staged_q = h->ws.staged_q;
    a.staged_s = h->ws.staged_s;
    a.wscale = h->wkv_scale;
    a.hidden = static_cast<const uint16_t*>(hidden);
    a.hs_t = hs[0];
    a.hs_h = hs[1];
    a.out = static_cast<uint16_t*>(out);
    a.os_t = os[0];
    a.os_h = os[1];
    a.mask = mask;
    a.qk = h->ws.qk;
    a.wpack = h->ws.wpack;
    a.part = h->ws.fpart;
    a.value = h->ws.fvalue;
    a.bar = h->ws.grid_bar;
    a.gate_out = h->ws.gate;
    a.eps = static_cast<float>(h->cfg.eps);
    a.clamp = static_cast<float>(h->cfg.clamp);
    a.inv_d = 1.0f / static_cast<float>(a.D);
    a.inv_sqrt_d = 1.0f / sqrtf(static_cast<float>(a.D));
    a.err = h->ws.err;
    // shared memory: stages | hidden rows | q*k slice | barriers; every stage
    // and its token tile 1024-byte aligned
    const int HR = a.T * a.H;
    const int rows_per_cta = (HR + p.grid - 1) / p.grid;
    const uint32_t row_bytes = static_cast<uint32_t>(a.D * 2);
    const uint32_t qk_bytes = kMaxFusedSlice * 4;
    const uint32_t bar_bytes = 512;
    a.w_stage_bytes = static_cast<uint32_t>((p.max_width * 128 + 1023) / 1024 * 1024);
    const uint32_t stage_bytes = a.w_stage_bytes + p.mtiles * 16384u;
    uint32_t hid_rows = static_cast<uint32_t>(rows_per_cta < kHidRows ? rows_per_cta : kHidRows);
    const uint32_t budget = kFusedSmemBytes - 1024;
    int stages = 0;
    for (;;) {
        const uint32_t fixed = hid_rows * row_bytes + qk_bytes + bar_bytes;
        stages = fixed < budget ? static_cast<int>((budget - fixed) / stage_bytes) : 0;
        if (stages >= 4 || hid_rows == 0) break;
        --hid_rows;
    }
    if (stages > kMaxStages) stages = kMaxStages;
    // the finish keeps each row's value and partial records in the stage buffers
    const int64_t fin_bytes =
        static_cast<int64_t>(rows_per_cta) * (a.D + p.grid * kPartFloats) * 4;
    if (stages < 2 || fin_bytes > static_cast<int64_t>(stages) * stage_bytes || rows_per_cta > 32)
        return cudaErrorInvalidConfiguration;
    a.stages = stages;
    a.hid_rows = hid_rows;
    a.hid_off = static_cast<uint32_t>(stages) * stage_bytes;
    a.qk_off = a.hid_off + hid_rows * row_bytes;
    a.bar_off = a.qk_off + qk_bytes;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kFusedSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const CUtensorMap* tmx = p.mtiles == 1 ? &h->tm_act_n[p.Tn / 16 - 1] : &h->tm_act_m;
    void* args[] = {const_cast<CUtensorMap*>(tmx), &a};
    const bool mx = h->cfg.wkv_format == ENGRAM_WKV_MXFP8;
    return cudaLaunchKernelExC(
        &cfg,
        mx ? reinterpret_cast<const void*>(decode_fused_kernel<true>)
           : reinterpret_cast<const void*>(decode_fused_kernel<false>),
        args);
}

}  // namespace engram
