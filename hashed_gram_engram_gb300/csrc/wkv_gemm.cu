// wkv projection on the fifth-generation tensor cores (tcgen05, TMEM
// accumulators, TMA-fed shared memory), sm_103a.
//
// kv = rows . wkv^T, rows = the staged gather output [T, K] (Engram.forward:
// wkv(embed(hash_ids).flatten(-2))), wkv [N, K] with N = D * (H + 1): keys
// h = 0..H-1 in columns [h*D, (h+1)*D), the shared value in [H*D, N)
// ("vllm.models.deepseek_v4_1.common.engram", Engram.__init__ and forward).
//
// This is the prefill schedule (T > 256; decode runs in decode_fused.cu):
// persistent clusters of two CTAs stride over units of 256 tokens x BN kv
// columns (BN = 256 for bf16), the pair sharing each MMA (see kPair below);
// where no pair cluster fits, single CTAs stride over 128-token tiles.
// The epilogue never writes keys: for a key tile it reduces
// (sum hidden^2, sum key^2, sum hidden*q*k*key) over the tile's dims -- the
// split-dim gate partials of _engram_gate_partials_kernel
// ("vllm.models.deepseek_v41.amd.engram"), here per N tile instead of per
// TP rank -- and for a value tile it stores the value in bf16.
//
// Roles: warp 0 = TMA producer, warp 1 = TMEM owner and (in a pair, the
// even CTA's only) MMA issuer, then
// the epilogue warps (TMEM lane quarter = warp % 4): 4 for bf16 (192
// threads); 8 for MXFP8 (320 threads, two per quarter taking half of the
// tile's columns each), whose short fp8 MMAs otherwise wait for the
// epilogue.  Two TMEM accumulators let the epilogue of one unit overlap the
// MMAs of the next.
// The weight loads of the first pipeline stages are issued before the
// programmatic-launch wait, overlapping the gather kernel.
//
// MXFP8 wkv: e4m3 codes of the rows (quantised by the gather) times e4m3
// weights, tcgen05 kind::mxf8f6f4 block_scale, 224 kv columns per unit when
// 224 divides dim (two accumulators of 224 columns and four 16-column scale
// slots fill the 512 TMEM columns), else 128.  Each stage also brings
// the 512-byte scale-factor atoms of its k-block (the tokens', and one per
// 128 tile rows of the weights', packed per tile at create); the MMA
// thread copies them into that stage's TMEM scale slot
// with tcgen05.cp right before the stage's MMAs.  A slot is rewritten only
// after the MMAs that read it have completed (the producer reuses a stage
// only after their commit), so one slot per stage suffices.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace engram {
namespace {

// producer, MMA issuer and 4 epilogue warps (8 for MXFP8, whose tiles' MMAs are short)
constexpr int threads_for(bool mx) { return mx ? 320 : 192; }
constexpr int kMaxStages = 8;
constexpr int kStageBudget = 192 * 1024;
constexpr uint32_t kTmemCols = 512;

struct GemmArgs {
    int m_tiles, n_tiles, k_blocks, total, T, kb128;
    int bn;       // MMA N: kv columns per tile
    int stages;
    uint32_t a_bytes, b_bytes;
    uint32_t idesc;
    int D, H, J;
    const uint16_t* hidden;
    int64_t hs_t, hs_h;
    const float* qk;
    float4* partials;
    uint16_t* value;
    const uint8_t* sfa;  // MXFP8: scale atoms of the staged codes
    const uint8_t* sfb;  // MXFP8: scale atoms of wkv
    unsigned* err;
    int hv8;  // hidden rows and strides 32-byte aligned: 32-byte loads
};

struct Unit {
    int m, n;
};

// Tiles of this CTA in order: blockIdx.x, blockIdx.x + gridDim.x, ...
// CTA pairs (kPair): the unit is 256 tokens x BN columns, pair k (CTAs 2k,
// 2k + 1, one cluster) takes units k, k + gridDim.x / 2, ..., and CTA rank r
// of the pair holds token tile 2i + r of unit (i, n).  When the token tiles
// are odd in number the last pair's second tile lies past T (rows the
// staging buffer holds, padded to 256; the epilogue skips them).
template <bool kPair>
struct Schedule {
    const GemmArgs& a;
    int64_t cur, end, step;
    int rank;
    __device__ explicit Schedule(const GemmArgs& args)
        : a(args),
          cur(kPair ? blockIdx.x >> 1 : blockIdx.x),
          end(static_cast<int64_t>(kPair ? (args.m_tiles + 1) / 2 : args.m_tiles) * args.n_tiles),
          step(kPair ? gridDim.x >> 1 : gridDim.x),
          rank(kPair ? static_cast<int>(blockIdx.x & 1u) : 0) {}
    __device__ bool next(Unit& u) {
        if (cur >= end) return false;
        const int mi = static_cast<int>(cur / a.n_tiles);
        u.m = kPair ? 2 * mi + rank : mi;
        u.n = static_cast<int>(cur % a.n_tiles);
        cur += step;
        return true;
    }
};

__device__ __forceinline__ void fail(int* abort_flag, unsigned* err) {
    *reinterpret_cast<volatile int*>(abort_flag) = 1;
    atomicOr(err, ENGRAM_DEVERR_TIMEOUT);
}

// kPair: CTA pairs of one cluster share each MMA (tcgen05 cta_group::2,
// M = 256): each CTA's shared memory holds its 128 token rows and half of
// the tile's BN weight rows (tmBh: boxes of BN/2 rows), so a CTA loads
// about 2/3 of the operand bytes of an unpaired 128 x BN tile for the same
// MMA work.  The even CTA issues the MMAs; its full barriers count both
// CTAs' copies; its commits reach both CTAs' empty and tfull barriers; both
// CTAs' epilogues release its tempty barriers.  MXFP8: each CTA also loads
// its token rows' scale atom and all BN weight rows' atoms (tmSA, tmSB:
// the atom arrays as rows of 512 bytes, so that the odd CTA's copies can
// complete on the even CTA's barrier), and the even CTA's tcgen05.cp moves
// each CTA's atoms into its own TMEM.
template <bool kMx, int BN, bool kPair>
__global__ void __launch_bounds__(threads_for(kMx), 1)
    wkv_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmSA,
                    const __grid_constant__ CUtensorMap tmSB, const GemmArgs a) {
    constexpr int G = kPair ? 2 : 1;  // tcgen05 CTA group
    constexpr int kKElems = kMx ? 128 : 64;  // k per 128-byte block
    constexpr uint32_t kBAtoms = (BN + 127) / 128;  // weight scale atoms per k-block
    constexpr uint32_t kAtoms = kMx ? 512u * (1u + kBAtoms) : 0u;  // scale atoms per stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t tx_bytes = a.a_bytes + a.b_bytes + kAtoms;  // copied per stage and CTA
    const uint32_t stage_bytes = (tx_bytes + 1023u) & ~1023u;   // stride: swizzle atoms stay aligned
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.stages * stage_bytes);
    uint64_t* empty = full + kMaxStages;
    uint64_t* tfull = empty + kMaxStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
    const volatile int* abort_v = abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = kPair ? (blockIdx.x & 1u) : 0u;  // rank in the 2-CTA cluster
    // an epilogue warp is done with an accumulator (pair: the even CTA's
    // barrier, which counts both CTAs' warps)
    auto release_acc = [](uint64_t* bar) {
        if constexpr (kPair)
            mbar_arrive_cluster(cluster_addr(bar, 0));
        else
            mbar_arrive(bar);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], (kPair ? 2 : 1) * (kMx ? 8 : 4));  // every epilogue warp (of the pair)
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(kPair ? &tmBh : &tmB);
    }
    // both CTAs' barriers are initialised before either signals the other's
    if constexpr (kPair) cluster_sync();
    if (warp == 1) {
        tmem_alloc<G>(tmem_slot, kTmemCols);
        tmem_relinquish<G>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    int64_t issued = 0;  // producer: pipeline iterations issued
    if (warp == 0) {
        if (lane == 0) {
            // The weight operand is independent of the gather; only the
            // token operand waits for the preceding kernel.
            const uint64_t pol_w = policy_evict_last();
            // token tile (and, MXFP8, its scale atom) of stage s
            auto load_x = [&](int s, int kb, int row) {
                uint8_t* sx = smem + s * stage_bytes;
                if constexpr (kPair)
                    tma_load_2d_pair(sx, &tmA, cluster_addr(&full[s], 0), kb * kKElems, row);
                else
                    tma_load_2d(sx, &tmA, &full[s], kb * kKElems, row);
                if constexpr (kMx && kPair)
                    tma_load_2d_pair(sx + a.a_bytes + a.b_bytes, &tmSA, cluster_addr(&full[s], 0), 0,
                                     (row / kBM) * a.kb128 + kb);
                else if constexpr (kMx)
                    bulk_load(sx + a.a_bytes + a.b_bytes,
                              a.sfa + (static_cast<int64_t>(row / kBM) * a.kb128 + kb) * 512, 512,
                              &full[s]);
            };
            Schedule<kPair> sch(a);
            Unit u;
            bool ok = true, waited = false;
            int pro_kb[kMaxStages], pro_row[kMaxStages], pro_s[kMaxStages];
            int npro = 0;
            int s = 0;         // stage of the next iteration
            uint32_t par = 0;  // its phase parity
            while (ok && sch.next(u)) {
                for (int kb = 0; kb < a.k_blocks; ++kb) {
                    if (!waited && issued == a.stages) {
                        // Every stage holds a weight tile: now wait for the
                        // gather and add the token tiles of those stages
                        // before any stage is recycled.
                        pdl_wait();
                        waited = true;
                        for (int i = 0; i < npro; ++i)
                            load_x(pro_s[i], pro_kb[i], pro_row[i]);
                    }
                    if (!mbar_wait(&empty[s], par ^ 1u, abort_v)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sw = smem + s * stage_bytes + a.a_bytes;
                    const int x_row = u.m * kBM;
                    if constexpr (kPair) {
                        // the even CTA's barrier counts both CTAs' bytes
                        if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * tx_bytes);
                        tma_load_2d_pair_hint(sw, &tmBh, cluster_addr(&full[s], 0), kb * kKElems,
                                              u.n * BN + static_cast<int>(rank) * (BN / 2), pol_w);
                    } else {
                        mbar_arrive_expect_tx(&full[s], tx_bytes);
                        tma_load_2d_hint(sw, &tmB, &full[s], kb * kKElems, u.n * BN, pol_w);
                    }
                    if constexpr (kMx && kPair)
                        tma_load_2d_pair(sw + a.b_bytes + 512, &tmSB, cluster_addr(&full[s], 0), 0,
                                         (u.n * a.kb128 + kb) * static_cast<int>(kBAtoms));
                    else if constexpr (kMx)
                        bulk_load(sw + a.b_bytes + 512,
                                  a.sfb + (static_cast<int64_t>(u.n) * a.kb128 + kb) * (512 * kBAtoms),
                                  512 * kBAtoms, &full[s]);
                    if (!waited) {
                        pro_kb[npro] = kb;
                        pro_row[npro] = x_row;
                        pro_s[npro] = s;
                        ++npro;
                    } else {
                        load_x(s, kb, x_row);
                    }
                    ++issued;
                    if (++s == a.stages) {
                        s = 0;
                        par ^= 1u;
                    }
                }
            }
            if (!waited) {
                pdl_wait();
                for (int i = 0; i < npro; ++i) load_x(pro_s[i], pro_kb[i], pro_row[i]);
            }
            pdl_launch_dependents();
            if (!ok) fail(abort_flag, a.err);
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {  // (a pair's odd CTA issues no MMA)
            Schedule<kPair> sch(a);
            Unit u;
            bool ok = true;
            int nu = 0;
            // The issuing thread's scalar latency sets the pace: the stage,
            // its parity, descriptors and scale slot advance incrementally
            // (a descriptor's address field is the byte address / 16).
            int s = 0;
            uint32_t par = 0;
            const uint32_t sa0 = smem_addr(smem);
            const uint64_t adesc0 = smem_desc_sw128(sa0);
            const uint64_t bdesc0 = smem_desc_sw128(sa0 + a.a_bytes);
            const uint64_t dstep = stage_bytes >> 4;
            uint32_t sa = sa0;
            uint64_t adesc = adesc0, bdesc = bdesc0;
            uint32_t sf = tmem_base + 2u * BN;  // MXFP8: this stage's scale slot
            while (ok && sch.next(u)) {
                const int acc = nu & 1;
                const uint32_t apar = static_cast<uint32_t>((nu >> 1) & 1);
                if (!mbar_wait(&tempty[acc], apar ^ 1u, abort_v, kPair)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < a.k_blocks; ++kb) {
                    if (!mbar_wait(&full[s], par, abort_v)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if constexpr (kMx) {
                        // this stage's 16-column scale slot: tokens' cells at
                        // +0, wkv's at +8 (4 columns per 128 tile rows)
                        const uint32_t atoms = sa + a.a_bytes + a.b_bytes;
                        if constexpr (kPair) {
                            tmem_cp_atom_pair(sf, smem_desc_atom(atoms));
#pragma unroll
                            for (uint32_t b = 0; b < kBAtoms; ++b)
                                tmem_cp_atom_pair(sf + 8 + 4 * b,
                                                  smem_desc_atom(atoms + 512 * (1 + b)));
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                mma_mxf8_ss_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k,
                                                 idesc_mxf8(2 * kBM, BN, k, k), sf, sf + 8,
                                                 (kb > 0 || k > 0) ? 1u : 0u);
                        } else {
                            tmem_cp_atom(sf, smem_desc_atom(atoms));
#pragma unroll
                            for (uint32_t b = 0; b < kBAtoms; ++b)
                                tmem_cp_atom(sf + 8 + 4 * b, smem_desc_atom(atoms + 512 * (1 + b)));
#pragma unroll
                            for (int k = 0; k < 4; ++k)  // 4 x K32, scale byte k of each cell
                                mma_mxf8_ss(d_tmem, adesc + 2 * k, bdesc + 2 * k,
                                            idesc_mxf8(kBM, BN, k, k), sf, sf + 8,
                                            (kb > 0 || k > 0) ? 1u : 0u);
                        }
                    } else if constexpr (kPair) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_bf16_ss_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, a.idesc,
                                             (kb > 0 || k > 0) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int k = 0; k < 4; ++k)  // 4 x K16 per 64-element block
                            mma_bf16_ss(d_tmem, adesc + 2 * k, bdesc + 2 * k, a.idesc,
                                        (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    if constexpr (kPair)
                        mma_commit_pair_mc(&empty[s], static_cast<uint16_t>(3));
                    else
                        mma_commit(&empty[s]);
                    if (++s == a.stages) {
                        s = 0;
                        par ^= 1u;
                        sa = sa0;
                        adesc = adesc0;
                        bdesc = bdesc0;
                        sf = tmem_base + 2u * BN;
                    } else {
                        sa += stage_bytes;
                        adesc += dstep;
                        bdesc += dstep;
                        sf += 16u;
                    }
                }
                if (!ok) break;
                if constexpr (kPair)
                    mma_commit_pair_mc(&tfull[acc], static_cast<uint16_t>(3));
                else
                    mma_commit(&tfull[acc]);
                ++nu;
            }
            if (!ok) fail(abort_flag, a.err);
        }
    } else {
        // Epilogue: TMEM lane quarter q = warp % 4, one accumulator row per
        // thread.  MXFP8: two warps per quarter, each taking half of the
        // tile's 32-column chunks (an epilogue must keep up with one tile's
        // MMAs, short at fp8), each half writing its own partial record.
        const int q = warp & 3;
        const int row = q * 32 + lane;
        constexpr int kHalfCh = kMx ? (BN / 32 + 1) / 2 : BN / 32;  // chunks of this warp
        const int half = kMx ? (warp - 2) >> 2 : 0;
        const int c0 = half * kHalfCh * 32;          // first column of this warp's half
        Schedule<kPair> sch(a);
        Unit u;
        bool ok = true;
        int nu = 0;
        while (sch.next(u)) {
            const int acc = nu & 1;
            const uint32_t apar = static_cast<uint32_t>((nu >> 1) & 1);
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
            {
                const int t = u.m * kBM + row;
                const bool live = t < a.T;
                const int col0 = u.n * BN;
                const int h = col0 / a.D;
                const int d0 = col0 - h * a.D;
                if (h < a.H) {
                    uint4 hv[kHalfCh * 4];
                    const uint16_t* hp = a.hidden + t * a.hs_t + h * a.hs_h + d0 + c0;
                    if (a.hv8) {  // half the load instructions
#pragma unroll
                        for (int i = 0; i < kHalfCh * 4; i += 2) {
                            hv[i] = hv[i + 1] = make_uint4(0, 0, 0, 0);
                            if (live && c0 + 8 * i < BN) ld_nc_v8(hp + 8 * i, hv[i], hv[i + 1]);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < kHalfCh * 4; ++i)
                            hv[i] = (live && c0 + 8 * i < BN) ? ld_nc_v4(hp + 8 * i)
                                                              : make_uint4(0, 0, 0, 0);
                    }
                    if (!mbar_wait(&tfull[acc], apar, abort_v)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const float* qkp = a.qk + h * a.D + d0 + c0;
                    float shh = 0.f, skk = 0.f, shk = 0.f;
#pragma unroll
                    for (int cc = 0; cc < kHalfCh; ++cc) {
                        const int c = cc * 32;  // within this half
                        if (c0 + c >= BN) break;
                        uint32_t r[32];
                        tmem_ld32(taddr + c0 + c, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; j += 8) {
                            // eight q*k values in one 32-byte load (one address for
                            // the whole warp; 32-byte aligned: tiles start on 32 dims)
                            uint4 q0, q1;
                            ld_nc_v8(qkp + c + j, q0, q1);
                            const float qk[8] = {__uint_as_float(q0.x), __uint_as_float(q0.y),
                                                 __uint_as_float(q0.z), __uint_as_float(q0.w),
                                                 __uint_as_float(q1.x), __uint_as_float(q1.y),
                                                 __uint_as_float(q1.z), __uint_as_float(q1.w)};
                            const uint4 hw = hv[(c + j) / 8];
                            const uint32_t w[4] = {hw.x, hw.y, hw.z, hw.w};
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float key = __uint_as_float(r[j + i]);
                                const float x = (i & 1) ? bf16hi(w[i >> 1]) : bf16lo(w[i >> 1]);
                                shh = fmaf(x, x, shh);
                                skk = fmaf(key, key, skk);
                                shk = fmaf(x * qk[i], key, shk);
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) release_acc(&tempty[acc]);
                    if (live)  // (MXFP8: J = 2 records per tile, one per half)
                        a.partials[(static_cast<int64_t>(t) * a.H + h) * a.J +
                                   (kMx ? 2 * (d0 / BN) + half : d0 / BN)] =
                            make_float4(shh, skk, shk, 0.f);
                } else {
                    if (!mbar_wait(&tfull[acc], apar, abort_v)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint16_t* vp = a.value + static_cast<int64_t>(t) * a.D + d0;
#pragma unroll
                    for (int cc = 0; cc < kHalfCh; ++cc) {
                        const int c = c0 + cc * 32;
                        if (c >= BN) break;
                        uint32_t r[32];
                        tmem_ld32(taddr + c, r);
                        tmem_ld_wait();
                        if (live) {
#pragma unroll
                            for (int j = 0; j < 32; j += 8) {
                                uint4 o;
                                o.x = pack_bf16x2(__uint_as_float(r[j + 0]), __uint_as_float(r[j + 1]));
                                o.y = pack_bf16x2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                                o.z = pack_bf16x2(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5]));
                                o.w = pack_bf16x2(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7]));
                                st_v4(vp + c + j, o);
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) release_acc(&tempty[acc]);
                }
            }
            ++nu;
        }
        if (!ok) fail(abort_flag, a.err);
    }

    // Teardown.  After a failed wait, let in-flight copies and MMAs land
    // (bounded) before the shared memory and TMEM are released.
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (*abort_v) {
        if (warp == 0 && lane == 0) {
            if (rank == 0) {
                const int64_t first = issued > a.stages ? issued - a.stages : 0;
                for (int64_t j = first; j < issued; ++j)
                    mbar_wait(&full[j % a.stages], static_cast<uint32_t>((j / a.stages) & 1),
                              nullptr);
            } else {
                // a pair's odd CTA: its copies complete on the even CTA's
                // barriers; give them 100 us to land
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 100000ull) __nanosleep(1000);
            }
        }
        if (warp == 1 && lane == 0 && rank == 0) {
            if constexpr (kPair)
                mma_commit_pair(drain);
            else
                mma_commit(drain);
            mbar_wait(drain, 0, nullptr);
        }
        __syncthreads();
    } else if constexpr (kPair) {
        // The even CTA's commits of the last stages have reached this CTA's
        // empty barriers (none is in flight toward it when the pair leaves).
        if (warp == 0 && lane == 0) {
            const int64_t first = issued > a.stages ? issued - a.stages : 0;
            for (int64_t j = first; j < issued; ++j)
                mbar_wait(&empty[j % a.stages], static_cast<uint32_t>((j / a.stages) & 1),
                          nullptr);
        }
        __syncthreads();
    }
    // a pair leaves together: neither CTA's shared memory or TMEM goes while
    // the other may still signal, read or write it
    if constexpr (kPair) cluster_sync();
    if (warp == 1) tmem_dealloc<G>(tmem_base, kTmemCols);
}

// E8M0 [N/32][K/32] block scales of wkv -> atoms [N/bn][K/128][ceil(bn/128)][512]
// per prefill tile of bn rows (byte 16*i + 4*j + b of atom (tile, kb, a) =
// scale of tile row 128a + 32j + i, k-block 4kb + b; rows past the tile,
// which no MMA reads, get 2^0).
__global__ void pack_scale_atoms_kernel(const uint8_t* ws, uint8_t* atoms, int64_t N, int64_t K,
                                        int64_t bn) {
    const int64_t o = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t kb128 = K / 128, nb = (bn + 127) / 128;
    if (o >= (N / bn) * kb128 * nb * 512) return;
    const int64_t w = o & 511, atom = o >> 9;
    const int64_t a = atom % nb, tk = atom / nb;
    const int64_t tile = tk / kb128, kb = tk - tile * kb128;
    const int64_t r = 128 * a + 32 * ((w >> 2) & 3) + (w >> 4);
    const int64_t k32 = 4 * kb + (w & 3);
    atoms[o] = r < bn ? ws[((tile * bn + r) >> 5) * (K >> 5) + k32] : static_cast<uint8_t>(127);
}

// Staged MXFP8 scale atoms -> plain [T][K/32], for validation.
__global__ void unpack_scale_atoms_kernel(const uint8_t* atoms, uint8_t* out, int64_t T,
                                          int64_t K) {
    const int64_t o = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (o >= T * (K / 32)) return;
    const int64_t t = o / (K / 32), k32 = o - t * (K / 32);
    out[o] = atoms[sf_atom_offset(t, k32, K / 128)];
}

}  // namespace

cudaError_t pack_scale_atoms(const engram_handle* h, cudaStream_t s) {
    const int64_t bn = prefill_bn(h);
    const int64_t n = (h->N / bn) * ((bn + 127) / 128) * (h->K / 128) * 512;
    pack_scale_atoms_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(
        h->wkv_scale, h->ws.wsf_atoms, h->N, h->K, bn);
    return cudaGetLastError();
}

cudaError_t launch_unpack_scales(const engram_handle* h, uint8_t* out, int64_t T,
                                 cudaStream_t s) {
    const int64_t n = T * (h->K / 32);
    unpack_scale_atoms_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(
        h->ws.staged_s, out, T, h->K);
    return cudaGetLastError();
}

// The kernel of a configuration: bf16 or MXFP8 weights, tile width, pairs.
static const void* gemm_kernel(bool mx, int bn, bool pair) {
    if (!mx)
        return pair ? reinterpret_cast<const void*>(wkv_gemm_kernel<false, kBNPrefill, true>)
                    : reinterpret_cast<const void*>(wkv_gemm_kernel<false, kBNPrefill, false>);
    if (bn == kBNPrefillMxWide)
        return pair ? reinterpret_cast<const void*>(wkv_gemm_kernel<true, kBNPrefillMxWide, true>)
                    : reinterpret_cast<const void*>(wkv_gemm_kernel<true, kBNPrefillMxWide, false>);
    return pair ? reinterpret_cast<const void*>(wkv_gemm_kernel<true, kBNPrefillMx, true>)
                : reinterpret_cast<const void*>(wkv_gemm_kernel<true, kBNPrefillMx, false>);
}

cudaError_t gemm_setup_attributes() {
    for (int mx = 0; mx < 2; ++mx)
        for (int pair = 0; pair < 2; ++pair)
            for (int bn : {kBNPrefillMx, kBNPrefillMxWide}) {
                const cudaError_t e =
                    cudaFuncSetAttribute(gemm_kernel(mx != 0, bn, pair != 0),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmemBytes);
                if (e != cudaSuccess) return e;
            }
    return cudaSuccess;
}

static cudaError_t launch(const void* fn, int grid, int threads, uint32_t smem_bytes, bool pair,
                          const engram_handle* h, const GemmArgs& a, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (pair) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 2;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    void* args[] = {const_cast<CUtensorMap*>(&h->tm_act_m), const_cast<CUtensorMap*>(&h->tm_w_n),
                    const_cast<CUtensorMap*>(&h->tm_w_half), const_cast<CUtensorMap*>(&h->tm_sfa),
                    const_cast<CUtensorMap*>(&h->tm_sfb), const_cast<GemmArgs*>(&a)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// Pipeline shape of a configuration: bytes per stage (a CTA's token rows,
// its weight rows -- half the tile's in a pair -- and, MXFP8, the scale
// atoms, rounded to 1024) and the number of stages (MXFP8: two accumulators
// plus a 16-column scale slot per stage in TMEM).
struct Pipe {
    uint32_t a_bytes, b_bytes, stride;
    int stages;
};

static Pipe pipe_shape(bool mx, int bn, bool pair) {
    Pipe p;
    p.a_bytes = kBM * kKBlockBytes;
    p.b_bytes = static_cast<uint32_t>(pair ? bn / 2 : bn) * kKBlockBytes;
    const uint32_t atoms = mx ? 512u * (1u + static_cast<uint32_t>((bn + 127) / 128)) : 0u;
    p.stride = (p.a_bytes + p.b_bytes + atoms + 1023u) & ~1023u;
    p.stages = static_cast<int>(kStageBudget / p.stride);
    if (p.stages > kMaxStages) p.stages = kMaxStages;
    if (mx && p.stages > (512 - 2 * bn) / 16) p.stages = (512 - 2 * bn) / 16;
    return p;
}

// the shared memory the stages and barriers need, and no more: the
// epilogue's loads go through the L1 that shares the SM's memory
static uint32_t smem_request(const Pipe& p) {
    return static_cast<uint32_t>(p.stages) * p.stride + 2048u;
}

// How many CTA-pair clusters of this configuration's GEMM fit on the GPU at
// once (0: none; the GEMM then runs on single CTAs).
int gemm_pair_capacity(const engram_handle* h) {
    const bool mx = h->cfg.wkv_format == ENGRAM_WKV_MXFP8;
    const int bn = prefill_bn(h);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * (h->num_sms / 2)));
    cfg.blockDim = dim3(static_cast<unsigned>(threads_for(mx)));
    cfg.dynamicSmemBytes = smem_request(pipe_shape(mx, bn, true));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, gemm_kernel(mx, bn, true), &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return clusters;
}

int prefill_bn(const engram_handle* h) {
    if (h->cfg.wkv_format != ENGRAM_WKV_MXFP8) return kBNPrefill;
    // The widest MXFP8 tile whose two accumulators and the stages' scale
    // slots fit TMEM, when it divides dim (then it divides N too).
    return h->cfg.dim % kBNPrefillMxWide == 0 ? kBNPrefillMxWide : kBNPrefillMx;
}

cudaError_t launch_wkv_tokens_m(const engram_handle* h, const void* hidden, int64_t hs_t,
                                int64_t hs_h, int64_t T, cudaStream_t s, bool pdl) {
    const bool mx = h->cfg.wkv_format == ENGRAM_WKV_MXFP8;
    const int bn = prefill_bn(h);
    // CTA pairs (256-token units, each CTA loading half the weight rows)
    // whenever their clusters fit
    const bool pair = h->gemm_pair_clusters > 0;
    const Pipe p = pipe_shape(mx, bn, pair);
    GemmArgs a = {};
    a.m_tiles = static_cast<int>((T + kBM - 1) / kBM);
    a.n_tiles = static_cast<int>(h->N / bn);
    a.k_blocks = static_cast<int>(h->K * (mx ? 1 : 2) / kKBlockBytes);
    a.kb128 = static_cast<int>(h->K / 128);
    a.total = a.m_tiles * a.n_tiles;
    a.T = static_cast<int>(T);
    a.bn = bn;
    a.a_bytes = p.a_bytes;
    a.b_bytes = p.b_bytes;
    a.stages = p.stages;
    a.idesc = idesc_bf16(pair ? 2 * kBM : kBM, kBNPrefill);  // bf16 only: MXFP8 builds one per k step
    a.D = static_cast<int>(h->cfg.dim);
    a.H = static_cast<int>(h->cfg.hc_mult);
    a.J = (mx ? 2 : 1) * (a.D / bn);  // MXFP8: a partial record per half tile
    a.hidden = static_cast<const uint16_t*>(hidden);
    a.hs_t = hs_t;
    a.hs_h = hs_h;
    // tile starts are multiples of 128 dims, so rows at 32-byte aligned
    // addresses keep every 32-byte load aligned
    a.hv8 = (reinterpret_cast<uintptr_t>(hidden) % 32 == 0 && hs_t % 16 == 0 && hs_h % 16 == 0)
                ? 1 : 0;
    a.qk = h->ws.qk;
    a.partials = h->ws.partials;
    a.value = h->ws.value;
    a.sfa = h->ws.staged_s;
    a.sfb = h->ws.wsf_atoms;
    a.err = h->ws.err;
    int grid;
    if (pair) {
        const int units = ((a.m_tiles + 1) / 2) * a.n_tiles;
        grid = 2 * (units < h->gemm_pair_clusters ? units : h->gemm_pair_clusters);
    } else {
        grid = a.total < h->num_sms ? a.total : h->num_sms;
    }
    return launch(gemm_kernel(mx, bn, pair), grid, threads_for(mx), smem_request(p), pair, h, a, s,
                  pdl);
}

}  // namespace engram
