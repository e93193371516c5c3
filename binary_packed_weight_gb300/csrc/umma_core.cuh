// umma_core.cuh -- the tcgen05 GEMM core shared by the ternary TQ2 path and
// the binary low-rank (blr) layer:
//
//   D[t, n] = sum_k act[t, k] * P[n, k]
//
// P is a packed plane (2-bit ternary codes with f16 block scales, or 1-bit
// signs) decoded on chip; act is an f16 activation matrix staged in the K
// order the decoder emits pairs in.  One CTA computes a 128 (plane rows) x BN
// (tokens) tile:
//   * eight decoder warps (one plane row per thread, two warps per row
//     quarter taking alternate K stages) write the decoded f16 rows into a
//     shared-memory ring in the MMA's K-major 128-byte-swizzled layout, so
//     tensor memory holds only the two accumulators;
//   * one thread issues TMA loads of the activation tile (B operand, 128-byte
//     swizzle) into a 4-stage shared-memory ring;
//   * one thread issues tcgen05.mma (kind::f16, f32 accumulate in TMEM) into
//     one of two accumulators and frees stages with tcgen05.commit;
//   * four epilogue warps read the finished accumulator (tcgen05.ld), hand it
//     back, and run the epilogue policy of the call while the next tile's
//     MMAs proceed in the other accumulator.
// All waits are bounded (mbar_wait); a timeout records an error and drains.
#pragma once

#include "ptx.cuh"
#include "tq2_internal.h"

namespace tq2 {

constexpr int UM_BM = 128;       // plane rows per tile = MMA M
constexpr int UM_BK = 64;        // K per pipeline stage (128 bytes of f16)
constexpr int UM_STAGES = 8;     // ring slots allocated; the launch picks how many it uses
constexpr int UM_MAX_BN = 256;   // MMA N limit for M = 128
constexpr int UM_A_STAGE = UM_BM * UM_BK * 2;   // decoded weight stage in shared memory (16 KB)
// warp 0 TMA, warp 1 MMA, warp 2 TMEM allocator, warp 3 idle,
// warps 4-11 decoders (two per 32-row quarter of the tile, taking alternate stages),
// warps 12-15 epilogue (one per lane quarter)
constexpr int UM_THREADS = 512;

struct UmmaBars {
    uint64_t full_b[UM_STAGES];
    uint64_t full_a[UM_STAGES];
    uint64_t empty[UM_STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ uint4 ldg_u4_nc(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ldg_u2_nc(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// ---------------------------------------------------------------- decoders ----
// A decoder turns K-stage kc (64 elements) of plane row `row` (valid iff ok)
// into 32 f16 pairs v[0..31]: pair j of the row holds K positions 2j, 2j+1 of
// the permuted order the activations are staged in (16-byte chunk j/4 of the
// row's 128 bytes, before the swizzle).  Loads go
// through L1 (the neighbouring stage of the same 32-byte sector is read by
// the partner decoder warp).

__device__ __forceinline__ uint4 ldg_u4_l1(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ldg_u2_l1(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// TQ2 codes: 16 bytes (four 16-element words) per stage, element e of a word
// at bits 2e; pair q = (element q, element q+8); the block scale is folded
// in: (c-1)*d is exact in f16.  Activations staged in 16-element groups.
struct DecTQ2 {
    const uint8_t* codes;      // [rows][K/4]
    const uint16_t* scales;    // [rows][K/128]
    int64_t pitch;             // K/4
    int nb;                    // K/128
    static constexpr int PF = 3;   // stages each decoder warp loads ahead
    static constexpr bool PRIOR = false;   // rows written by earlier work on the stream (wait for it)
    struct Raw { uint4 c; uint16_t d; };
    __device__ __forceinline__ Raw load(int row, bool ok, int kc) const {
        Raw r;
        if (ok) {
            r.c = ldg_u4_l1(codes + (int64_t)row * pitch + (int64_t)kc * 16);
            r.d = __ldg(scales + (int64_t)row * nb + kc / 2);
        } else {
            r.c = make_uint4(0u, 0u, 0u, 0u);
            r.d = 0;
        }
        return r;
    }
    __device__ __forceinline__ void decode(const Raw& r, uint32_t (&v)[32]) const {
        const __half2 d2 = __halves2half2(__ushort_as_half(r.d), __ushort_as_half(r.d));
        const uint32_t words[4] = {r.c.x, r.c.y, r.c.z, r.c.w};
        uint32_t p[8];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            decode_word(words[w], p);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                __half2 hh = __hmul2(*reinterpret_cast<__half2*>(&p[q]), d2);
                v[w * 8 + q] = *reinterpret_cast<uint32_t*>(&hh);
            }
        }
    }
};

// Sign bits: two 32-sign words per stage (bit b = element b of a word, set =
// +1); pair p = (element p, element p+16).  Activations staged in 32-element
// groups.
struct DecSign {
    const uint32_t* bits;      // [rows][K/32]
    int64_t words;             // K/32
    static constexpr int PF = 3;
    static constexpr bool PRIOR = true;    // the caller's bitmaps may come from the kernel before
    struct Raw { uint2 w; };
    __device__ __forceinline__ Raw load(int row, bool ok, int kc) const {
        Raw r;
        r.w = ok ? ldg_u2_l1(bits + (int64_t)row * words + (int64_t)kc * 2) : make_uint2(0u, 0u);
        return r;
    }
    template <int P>
    __device__ __forceinline__ static uint32_t pair(uint32_t w) {
        // bit P -> bit 15, bit P+16 -> bit 31; set bit -> +1 (0x3C00), clear -> -1 (0xBC00)
        return ((w << (15 - P)) & 0x80008000u) ^ 0xBC00BC00u;
    }
    __device__ __forceinline__ static void word(uint32_t w, uint32_t* o) {
        o[0] = pair<0>(w);   o[1] = pair<1>(w);   o[2] = pair<2>(w);   o[3] = pair<3>(w);
        o[4] = pair<4>(w);   o[5] = pair<5>(w);   o[6] = pair<6>(w);   o[7] = pair<7>(w);
        o[8] = pair<8>(w);   o[9] = pair<9>(w);   o[10] = pair<10>(w); o[11] = pair<11>(w);
        o[12] = pair<12>(w); o[13] = pair<13>(w); o[14] = pair<14>(w); o[15] = pair<15>(w);
    }
    __device__ __forceinline__ void decode(const Raw& r, uint32_t (&v)[32]) const {
        word(r.w.x, v);
        word(r.w.y, v + 16);
    }
};

// Dense f16 rows, already in the K order the activations are staged in
// (pair j of a stage = elements 2j, 2j+1): the decoder only moves them.  A
// stage is 128 bytes per row, so one stage is loaded ahead.
struct DecDense {
    const uint16_t* rows;      // [rows][pitch] f16 bits
    int64_t pitch;             // elements per row (a multiple of 64)
    static constexpr int PF = 1;
    static constexpr bool PRIOR = true;    // staged by the kernel before this one
    struct Raw { uint4 q[8]; };
    __device__ __forceinline__ Raw load(int row, bool ok, int kc) const {
        Raw r;
        const uint4* src = reinterpret_cast<const uint4*>(rows + (int64_t)row * pitch + (int64_t)kc * 64);
#pragma unroll
        for (int i = 0; i < 8; ++i) r.q[i] = ok ? ldg_u4_l1(src + i) : make_uint4(0u, 0u, 0u, 0u);
        return r;
    }
    __device__ __forceinline__ void decode(const Raw& r, uint32_t (&v)[32]) const {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[4 * i] = r.q[i].x;
            v[4 * i + 1] = r.q[i].y;
            v[4 * i + 2] = r.q[i].z;
            v[4 * i + 3] = r.q[i].w;
        }
    }
};

// --------------------------------------------------------------- epilogues ----
enum EpiMode : int {
    EPI_STORE = 0,        // out[t][n] = acc * oscale
    EPI_ATOMIC = 1,       // out[t][n] += acc * oscale (atomic; two K splits at most)
    EPI_SCALE = 3,        // out[t][n] (+)= acc * oscale * vec[n]; out2[t][n] = acc * oscale if out2
    EPI_SCALE_COLSUM = 4, // as EPI_SCALE, plus colpart[tile][n] = sum_t acc*oscale*other[t][n]
    EPI_COLSUM = 5        // colpart[tile][n] = sum_t acc*oscale*other[t][n] only
};

struct EpiArgs {
    float* out;
    float* out2;
    const float* vec;
    const float* other;
    float* colpart;        // [token tiles][ldo]
    int64_t ldo;           // row stride of out / out2 / other (= plane rows)
    float oscale;
    int accumulate;        // EPI_SCALE*: out = fl(out + fl(w * vec)) instead of fl(w * vec)
};

// ----------------------------------------------------------------- kernel ----
// Persistent: CTA b walks tiles b, b + gridDim.x, ...; tile t = (n-tile, token
// tile, K split) with the n-tile fastest, so CTAs running together share one
// activation tile in L2.  The stage ring and the two accumulators run
// continuously across tiles; the epilogue of a tile overlaps the MMAs of the
// next.
struct TileMap {
    // a unit is `cl` weight tiles (one per CTA of a cluster) x one token tile
    // x one K split; tiles_np = ceil(tiles_n / cl) units along the rows
    int tiles_n, tiles_np, tiles_m, splits, total, nk_total;
    __device__ __forceinline__ void decode(int t, int& np, int& m, int& z) const {
        np = t % tiles_np;
        const int rest = t / tiles_np;
        m = rest % tiles_m;
        z = rest / tiles_m;
    }
    __device__ __forceinline__ int kc0(int z) const { return (int)(((int64_t)nk_total * z) / splits); }
    __device__ __forceinline__ int kc1(int z) const { return (int)(((int64_t)nk_total * (z + 1)) / splits); }
};

// AT: the decoded weights go to tensor memory (an S-stage ring of 32
// columns a stage after the NACC accumulators) instead of shared memory, and
// the MMAs read A from there; for token tiles of at most 128, where the
// shared-memory round trip of the decoded rows would cost more than the MMAs.
template <class Dec, int MODE, bool AT>
__global__ void __launch_bounds__(UM_THREADS, 1)
umma_gemm_kernel(const __grid_constant__ CUtensorMap xmap, const Dec dec, const EpiArgs ep, int T, int R, int BN,
                 int tmem_cols, const TileMap tm, int S, int NACC, int cl) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int stage_bytes = BN * 128;
    uint8_t* a_ring = smem + S * stage_bytes;            // [S][128 rows][128 B], swizzled; 1 KB aligned (!AT)
    UmmaBars* bars = reinterpret_cast<UmmaBars*>(a_ring + (AT ? 0 : S * UM_A_STAGE));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // cluster of cl CTAs (1 or 2): the CTAs of a cluster take adjacent weight
    // tiles of the same unit and share its activation tile: each loads 1/cl
    // of it with a multicast TMA into every CTA's ring.
    const int rank = cl > 1 ? (int)cluster_ctarank() : 0;
    const int unit0 = blockIdx.x / cl, units = gridDim.x / cl;
    const uint16_t cmask = (uint16_t)((1u << cl) - 1u);

    if (threadIdx.x == 0) {
        for (int s = 0; s < UM_STAGES; ++s) {
            mbar_init(&bars->full_b[s], 1);
            mbar_init(&bars->full_a[s], 4);
            mbar_init(&bars->empty[s], (uint32_t)cl);     // every cluster CTA's MMA must release it
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->acc_full[b], 1);
            mbar_init(&bars->acc_empty[b], 4);
        }
        bars->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&xmap);
    }
    if (warp == 2) {
        tmem_alloc(&bars->tmem_base, (uint32_t)tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    if (cl > 1) cluster_sync();                          // peers' barriers exist before any multicast
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t a_col0 = (uint32_t)(NACC * BN);       // first column of the A ring (AT)
    volatile int* abort_flag = &bars->abort;

    pdl_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {                                   // ---- TMA producer
            pdl_wait();
            int it = 0, s = 0;
            uint32_t ph = 0;                               // ring slot and phase parity of item `it`
            bool ok = true;
            for (int t = unit0; t < tm.total && ok && !*abort_flag; t += units) {
                int np, m, z;
                tm.decode(t, np, m, z);
                for (int kc = tm.kc0(z); kc < tm.kc1(z); ++kc, ++it) {
                    if (it >= S && !mbar_wait_or_abort(&bars->empty[s], ph ^ 1u, abort_flag)) {
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars->full_b[s], (uint32_t)stage_bytes);
                    const int part = BN / cl;                  // token rows this CTA loads
                    if (cl > 1)
                        tma_load_2d_mc(smem + s * stage_bytes + rank * part * 128, &xmap, &bars->full_b[s], kc * UM_BK,
                                       m * BN + rank * part, cmask);
                    else
                        tma_load_2d(smem + s * stage_bytes, &xmap, &bars->full_b[s], kc * UM_BK, m * BN);
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
            }
            // let the copies already issued land before the CTA can exit
            for (int i = (it > S ? it - S : 0); i < it; ++i)
                mbar_wait(&bars->full_b[i % S], (uint32_t)(i / S) & 1u);
        }
    } else if (warp == 1) {
        // ---- MMA issuer: the whole warp runs the loop, lane 0 waits on the
        // barriers, and every MMA and commit is issued by one lane chosen with
        // elect.sync, so the warp stays converged around the tcgen05 issue.
        const uint32_t idesc = idesc_f16_f32(UM_BM, (uint32_t)BN);
        int lt = 0, s = 0;
        uint32_t ph = 0;
        bool ok = true;
        auto wait1 = [&](uint64_t* bar, uint32_t parity) -> bool {
            int r = 1;
            if (lane == 0) r = mbar_wait_or_abort(bar, parity, abort_flag, true) ? 1 : 0;
            return __shfl_sync(0xffffffffu, r, 0) != 0;
        };
        for (int t = unit0; t < tm.total && ok; t += units, ++lt) {
            int np, m, z;
            tm.decode(t, np, m, z);
            const int buf = NACC == 2 ? (lt & 1) : 0, use = NACC == 2 ? (lt >> 1) : lt;
            if (use >= 1 && !wait1(&bars->acc_empty[buf], (uint32_t)(use - 1) & 1u)) {
                if (lane == 0) *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const uint32_t dcol = tmem + (uint32_t)(buf * BN);
            const int k0 = tm.kc0(z), k1 = tm.kc1(z);
            for (int kc = k0; kc < k1; ++kc) {
                if (!wait1(&bars->full_b[s], ph) || !wait1(&bars->full_a[s], ph)) {
                    if (lane == 0) *abort_flag = 1;
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(smem + s * stage_bytes));
                if (AT) {
                    const uint32_t acol = tmem + a_col0 + (uint32_t)(s * (UM_BK / 2));
#pragma unroll
                    for (int j = 0; j < UM_BK / 16; ++j)
                        umma_f16_ts_elect(dcol, acol + (uint32_t)(j * 8), bdesc + (uint64_t)(2 * j), idesc,
                                          (kc > k0 || j > 0) ? 1u : 0u);
                } else {
                    const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(a_ring + s * UM_A_STAGE));
#pragma unroll
                    for (int j = 0; j < UM_BK / 16; ++j)
                        umma_f16_ss_elect(dcol, adesc + (uint64_t)(2 * j), bdesc + (uint64_t)(2 * j), idesc,
                                          (kc > k0 || j > 0) ? 1u : 0u);
                }
                if (cl > 1) umma_commit_mc_elect(&bars->empty[s], cmask);
                else umma_commit_elect(&bars->empty[s]);
                if (++s == S) { s = 0; ph ^= 1u; }
            }
            if (!ok) break;
            umma_commit_elect(&bars->acc_full[buf]);
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        }
    } else if (warp >= 4 && warp < 12) {                   // ---- decoders
        // warp pair (q, h): lane quarter q, stages with item parity h
        const int q = warp & 3, h = (warp - 4) >> 2;
        const int arow = q * 32 + lane;                    // row of the A stage this thread writes
        constexpr int PF = Dec::PF;                        // own items prefetched ahead
        // flattened walk over this CTA's (tile, kc) items, two cursors
        struct Cur {
            int t, kc, k1, row;
            bool rok;
        };
        auto start = [&](Cur& c, int t) {
            c.t = t;
            if (t < tm.total) {
                int np, m, z;
                tm.decode(t, np, m, z);
                c.kc = tm.kc0(z);
                c.k1 = tm.kc1(z);
                c.row = (np * cl + rank) * UM_BM + q * 32 + lane;
                c.rok = c.row < R;
            }
        };
        auto step = [&](Cur& c) {
            if (++c.kc >= c.k1) start(c, c.t + units);
        };
        Cur ld, pr;
        if (Dec::PRIOR) pdl_wait();                        // the rows come from the previous kernel
        start(ld, unit0);
        start(pr, unit0);
        int ld_it = 0;
        typename Dec::Raw ring[PF];
        // advance the load cursor to this warp's first item and prefetch PF items
        auto next_own = [&](Cur& c, int& i) {
            while (c.t < tm.total && (i & 1) != h) { step(c); ++i; }
        };
        next_own(ld, ld_it);
#pragma unroll
        for (int j = 0; j < PF; ++j) {
            const bool live = ld.t < tm.total;
            ring[j] = dec.load(live && ld.rok ? ld.row : 0, live && ld.rok, live ? ld.kc : 0);
            if (live) { step(ld); ++ld_it; next_own(ld, ld_it); }
        }
        int it = 0, slot = 0, s = 0;
        uint32_t ph = 0;                                   // ring slot and phase parity of item `it`
        bool ok = true;
        while (pr.t < tm.total && ok) {
            if ((it & 1) == h) {
                const typename Dec::Raw cur = ring[0];
#pragma unroll
                for (int j = 0; j + 1 < PF; ++j) ring[j] = ring[j + 1];
                {
                    const bool live = ld.t < tm.total;
                    ring[PF - 1] = dec.load(live && ld.rok ? ld.row : 0, live && ld.rok, live ? ld.kc : 0);
                    if (live) { step(ld); ++ld_it; next_own(ld, ld_it); }
                }
                if (it >= S && !mbar_wait_or_abort(&bars->empty[s], ph ^ 1u, abort_flag)) {
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                uint32_t v[32];
                dec.decode(cur, v);
                if (AT) {
                    // row arow = TMEM lane arow; pair j of the stage in column j of the stage's 32
                    tc_fence_after();
                    tmem_st_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + a_col0 + (uint32_t)(s * (UM_BK / 2)), v);
                    tmem_wait_st();
                    tc_fence_before();
                } else {
                    // row arow of the stage: 16-byte chunk c (columns 4c..4c+3) at
                    // chunk c ^ (arow & 7), the layout TMA would write with 128-byte swizzle
                    uint8_t* rowp = a_ring + s * UM_A_STAGE + arow * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(rowp + ((c ^ (arow & 7)) << 4)) =
                            make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                    fence_proxy_async_shared();            // the MMA reads A through the async proxy
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->full_a[s]);
            }
            step(pr);
            ++it;
            if (++s == S) { s = 0; ph ^= 1u; }
            (void)slot;
        }
    } else if (warp >= 12) {                               // ---- epilogue
        const int q = warp & 3;
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        bool waited = false;
        int lt = 0;
        for (int t = unit0; t < tm.total; t += units, ++lt) {
            int np, m, z;
            tm.decode(t, np, m, z);
            const int n = np * cl + rank;
            const int buf = NACC == 2 ? (lt & 1) : 0, use = NACC == 2 ? (lt >> 1) : lt;
            if (!mbar_wait_or_abort(&bars->acc_full[buf], (uint32_t)use & 1u, abort_flag)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            if (!waited) {
                pdl_wait();
                waited = true;
            }
            const int row = n * UM_BM + q * 32 + lane;
            const bool rok = row < R;
            const int m0 = m * BN;
            const float vs = (rok && (MODE == EPI_SCALE || MODE == EPI_SCALE_COLSUM)) ? ep.vec[row] : 1.f;
            float colacc = 0.f;
            for (int cc = 0; cc < BN; cc += 32) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(lane_addr + (uint32_t)(buf * BN + cc), v);
                tmem_wait_ld();
                if (cc + 32 >= BN) {                       // accumulator fully read: hand it back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->acc_empty[buf]);
                }
                if (!rok) continue;
                const int nvalid = (T - (m0 + cc)) < 32 ? (T - (m0 + cc)) : 32;
                const int64_t o0 = (int64_t)(m0 + cc) * ep.ldo + row;
                auto one = [&](int i) {
                    const float a = __uint_as_float(v[i]);
                    const int64_t o = o0 + (int64_t)i * ep.ldo;
                    if (MODE == EPI_STORE) {
                        ep.out[o] = a * ep.oscale;
                    } else if (MODE == EPI_ATOMIC) {
                        atomicAdd(ep.out + o, a * ep.oscale);
                    } else {
                        const float w = a * ep.oscale;
                        if (MODE == EPI_SCALE || MODE == EPI_SCALE_COLSUM) {
                            // product and sum rounded separately (no fused multiply-add):
                            // the rounding of the pages' multi-path combine
                            const float pv = __fmul_rn(w, vs);
                            ep.out[o] = ep.accumulate ? __fadd_rn(ep.out[o], pv) : pv;
                            if (MODE == EPI_SCALE && ep.out2) ep.out2[o] = w;
                        }
                        if (MODE == EPI_SCALE_COLSUM || MODE == EPI_COLSUM) colacc = fmaf(w, ep.other[o], colacc);
                    }
                };
                if (nvalid == 32) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) one(i);
                } else {
                    for (int i = 0; i < nvalid; ++i) one(i);
                }
            }
            if ((MODE == EPI_SCALE_COLSUM || MODE == EPI_COLSUM) && rok)
                ep.colpart[(int64_t)m * ep.ldo + row] = colacc;
        }
    }

    tc_fence_before();
    __syncthreads();
    // every MMA of this CTA has completed (the epilogue saw each tile), so its
    // multicast commits have landed; wait for the peers' to land here too
    if (cl > 1) cluster_sync();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)tmem_cols);
    }
}

// Host: launch one GEMM.  act16 is f16 [T][K] (row pitch K), staged in the
// decoder's K order; R = plane rows; splits = K splits.  Token tiles of at
// most 128 keep the decoded weights in tensor memory (AT) and run without
// clusters; wider tiles decode into shared memory and pair CTAs on
// neighbouring weight tiles to share the activation tile.
template <class Dec, int MODE>
cudaError_t launch_umma(const Dec& dec, const EpiArgs& ep, const void* act16, int T, int R, int K, int BN, int splits,
                        cudaStream_t st);

template <class Dec, int MODE, bool AT>
cudaError_t launch_umma_impl(const Dec& dec, const EpiArgs& ep, const void* act16, int T, int R, int K, int BN,
                             int splits, cudaStream_t st) {
    if (BN > UM_MAX_BN || BN % 16 != 0 || BN < 16 || (AT && BN > 128)) return cudaErrorInvalidValue;
    // the epilogue drains 32 columns at a time: a tile narrower than a
    // multiple of 32 must be the only token tile
    if (BN % 32 != 0 && T > BN) return cudaErrorInvalidValue;
    const int tiles_n = (R + UM_BM - 1) / UM_BM;
    const int cl = (!AT && tiles_n >= 2 && BN % 32 == 0) ? 2 : 1;   // pairs share activation tiles
    CUtensorMap xmap;
    if (!make_tensor_map_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, const_cast<void*>(act16), (uint64_t)K,
                            (uint64_t)T, (uint64_t)K * 2, UM_BK, (uint32_t)(BN / cl), CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    // two accumulators in tensor memory (the epilogue of a tile overlaps the
    // next tile's MMAs); the B ring (and the A ring unless AT) fills the
    // shared memory; with AT the A ring takes S x 32 tensor-memory columns
    // after the accumulators (2 x 128 + 8 x 32 = 512 at most)
    const int NACC = 2;
    const int a_stage = AT ? 0 : UM_A_STAGE;
    int S = UM_STAGES;
    while (S > 2 && (size_t)S * (BN * 128 + a_stage) + sizeof(UmmaBars) + 1024 > (size_t)220 * 1024) --S;
    int tmem_cols = 32;
    while (tmem_cols < NACC * BN + (AT ? S * (UM_BK / 2) : 0)) tmem_cols <<= 1;
    if (tmem_cols > 512) return cudaErrorInvalidValue;
    // At least 120 KB of shared memory: no two CTAs of this kernel can share
    // an SM, so a CTA never waits in tcgen05.alloc for a co-resident CTA
    // (which a cluster barrier could otherwise turn into a deadlock).
    size_t smem = (size_t)S * (BN * 128 + a_stage) + 1024 + sizeof(UmmaBars) + 1024;
    if (smem < (size_t)120 * 1024) smem = (size_t)120 * 1024;
    TileMap tm;
    tm.tiles_n = tiles_n;
    tm.tiles_np = (tiles_n + cl - 1) / cl;
    tm.tiles_m = (T + BN - 1) / BN;
    tm.splits = splits;
    tm.total = tm.tiles_np * tm.tiles_m * splits;
    tm.nk_total = K / UM_BK;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int units = tm.total < sms / cl ? tm.total : sms / cl;
    cudaError_t e = cudaFuncSetAttribute(umma_gemm_kernel<Dec, MODE, AT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(units * cl));
    cfg.blockDim = dim3(UM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cl;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, umma_gemm_kernel<Dec, MODE, AT>, xmap, dec, ep, T, R, BN, tmem_cols, tm, S, NACC,
                              cl);
}

template <class Dec, int MODE>
cudaError_t launch_umma(const Dec& dec, const EpiArgs& ep, const void* act16, int T, int R, int K, int BN, int splits,
                        cudaStream_t st) {
    if (BN <= 128) return launch_umma_impl<Dec, MODE, true>(dec, ep, act16, T, R, K, BN, splits, st);
    return launch_umma_impl<Dec, MODE, false>(dec, ep, act16, T, R, K, BN, splits, st);
}

inline int umma_pick_bn(int T) {
    if (T >= 256) return 256;
    return ((T + 15) / 16) * 16;
}

}  // namespace tq2
