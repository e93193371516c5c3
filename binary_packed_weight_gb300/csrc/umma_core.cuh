// umma_core.cuh -- the tcgen05 GEMM core shared by the ternary TQ2 path and
// the binary low-rank (blr) layer:
//
//   D[t, n] = sum_k act[t, k] * P[n, k]
//
// P is a packed plane (2-bit ternary codes with f16 block scales, 1-bit
// signs) or dense f16 rows; act is an f16 activation matrix staged in the K
// order the decoder emits pairs in.  One CTA computes a 128 (plane rows) x BN
// (tokens) tile, in pipeline stages of KA x 64 k (KA = 4 for tiles of at
// most 128 tokens, 2 for the ternary GEMM's 256-token tiles, else 1):
//   * one thread streams the activation tiles (B operand, 128-byte swizzle)
//     into a ring of up to 8 stages with TMA;
//   * a second thread streams the packed plane tiles of the same stages (the
//     2-bit codes and block scales, or the sign words) with TMA into a
//     deeper ring of raw stages, far enough ahead to cover the HBM latency;
//     dense f16 rows skip the decoders: TMA writes them as the A operand;
//   * eight decoder warps (one plane row per thread, two warps per 32-row
//     quarter taking alternate stages) expand a raw stage from shared memory
//     into the f16 A operand: into tensor memory (AT: tiles of at most 128
//     tokens, the ternary GEMM's 256-token tiles and the 384-token wide
//     tile), otherwise into a shared-memory ring in the MMA's K-major
//     128-byte-swizzled layout;
//   * one warp issues tcgen05.mma (kind::f16, f32 accumulate in TMEM) into
//     one of two accumulators (one where A takes their room: 256 tokens with
//     AT and the wide tile) and frees stages with tcgen05.commit; every MMA
//     is issued by one lane of the converged warp (elect.sync);
//   * four epilogue warps read the finished accumulator (tcgen05.ld), hand it
//     back, and run the epilogue policy of the call while the next tile's
//     MMAs proceed in the other accumulator; for the column-sum policies of
//     short-K GEMMs the warp that allocated tensor memory streams their
//     operand in by TMA and the results go out by TMA store.
// Every CTA loads its own tiles (no clusters).
// All waits are bounded (mbar_wait); a timeout records an error and drains.
#pragma once

#include "ptx.cuh"
#include "tq2_internal.h"

namespace tq2 {

constexpr int UM_BM = 128;       // plane rows per tile = MMA M
constexpr int UM_BK = 64;        // K per pipeline stage (128 bytes of f16)
constexpr int UM_STAGES = 8;     // B / A ring slots allocated; the launch picks how many it uses
constexpr int UM_RAW_STAGES = 32;   // raw plane ring slots allocated
constexpr int UM_MAX_BN = 256;   // MMA N limit for M = 128
// The wide token tile: one 384-column accumulator and a 4-stage A ring in
// tensor memory fill its 512 columns, so a decoded stage feeds 384 tokens
// (two MMAs per k-step, N = 256 and 128) without a shared-memory A ring.
constexpr int UM_WIDE_BN = 384;
constexpr int UM_A_STAGE = UM_BM * UM_BK * 2;   // decoded weight stage in shared memory (16 KB)
// warp 0 activation TMA, warp 1 MMA, warp 2 TMEM allocator, warp 3 plane TMA,
// warps 4-11 decoders (two per 32-row quarter of the tile, taking alternate stages),
// warps 12-15 epilogue (one per lane quarter)
constexpr int UM_THREADS = 512;
// TMA epilogue: an input ring of UM_EPI_IN chunks of [32 tokens][128 rows]
// f32 (the column-sum operand), and per epilogue warp two output buffers of
// [32 tokens][32 rows] f32 stored by TMA
constexpr int UM_EPI_IN = 4;
constexpr int UM_EPI_IN_BYTES = 32 * UM_BM * 4;             // 16 KB
constexpr int UM_EPI_OUT_BYTES = 4 * 2 * 32 * 32 * 4;       // 32 KB
constexpr int UM_EPI_TMA_STEPS = 16;                        // K / 64 at most for the TMA epilogue

struct UmmaBars {
    uint64_t full[UM_STAGES];      // a stage's B tile landed (TMA bytes) and its A rows are decoded (4 warps)
    uint64_t empty[UM_STAGES];
    uint64_t raw_full[UM_RAW_STAGES];
    uint64_t raw_empty[UM_RAW_STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t epi_full[UM_EPI_IN];  // TMA epilogue: a 32-token chunk of the epilogue's input landed
    uint64_t epi_empty[UM_EPI_IN]; // ... and the four epilogue warps are done with it
    uint32_t tmem_base;
    int abort;
};

// ---------------------------------------------------------------- decoders ----
// A decoder describes the plane: RAW bytes a stage of its packed tile (TMA
// loads issued by issue()), and decode(), which turns row r (0..127) of a
// raw stage of K-stage kc (64 elements) into 32 f16 pairs v[0..31]: pair j
// holds K positions 2j, 2j+1 of the permuted order the activations are staged
// in (16-byte chunk j/4 of the row's 128 bytes, before the swizzle).
// DIRECT planes are already f16 in that order: TMA writes them as the A
// operand and no decoder runs.

// TQ2 codes: 16 bytes (four 16-element words) per row and stage, element e
// of a word at bits 2e; pair q = (element q, element q+8); the block scale is
// folded in: (c-1)*d is exact in f16.  Activations staged in 16-element
// groups.  Raw stage: codes [128 rows][16 B], then the stage's block scales
// [128 rows], both from the copies made at upload for this path (the codes
// stage-tiled, so a stage is 2 KB contiguous and lands as 16 lines of 128
// bytes; the scales block-major).  A 16-byte-wide box of the row-major plane
// streams at only about one row per 5 cycles.
struct DecTQ2 {
    static constexpr int RAW = UM_BM * 16 + UM_BM * 2;
    static constexpr bool DIRECT = false;
    __device__ __forceinline__ static void issue(const CUtensorMap* m0, const CUtensorMap* m1, uint8_t* raw,
                                                 uint64_t* bar, int row0, int kc) {
        tma_load_3d(raw, m0, bar, 0, kc * 16, row0 >> 7);     // codes: 16 lines of 128 B
        tma_load_2d(raw + UM_BM * 16, m1, bar, row0, kc / 2);   // scales: x = row, y = block
    }
    // a stage of KA = 2 or 4 atoms of 64 k (one or two blocks): codes
    // [KA][128 rows][16 B], then the blocks' scales [KA/2][128 rows]
    template <int KA>
    __host__ __device__ static constexpr int rawk() { return UM_BM * 16 * KA + UM_BM * 2 * (KA / 2); }
    template <int KA>
    __device__ __forceinline__ static void issuek(const CUtensorMap* m0, const CUtensorMap* m1, uint8_t* raw,
                                                  uint64_t* bar, int row0, int ks) {
#pragma unroll
        for (int p = 0; p < KA; ++p) tma_load_3d(raw + p * (UM_BM * 16), m0, bar, 0, (ks * KA + p) * 16, row0 >> 7);
#pragma unroll
        for (int b = 0; b < KA / 2; ++b)
            tma_load_2d(raw + KA * (UM_BM * 16) + b * (UM_BM * 2), m1, bar, row0, ks * (KA / 2) + b);
    }
    // atom p (k 64p .. 64p+63 of the stage) of row r
    template <int KA>
    __device__ __forceinline__ static void decodek(const uint8_t* raw, int r, int p, uint32_t (&v)[32]) {
        expand(*reinterpret_cast<const uint4*>(raw + p * (UM_BM * 16) + r * 16),
               reinterpret_cast<const uint16_t*>(raw + KA * (UM_BM * 16) + (p >> 1) * (UM_BM * 2))[r], v);
    }
    __device__ __forceinline__ static void decode(const uint8_t* raw, int r, int kc, uint32_t (&v)[32]) {
        expand(*reinterpret_cast<const uint4*>(raw + r * 16), reinterpret_cast<const uint16_t*>(raw + UM_BM * 16)[r],
               v);
        (void)kc;
    }
    __device__ __forceinline__ static void expand(const uint4 c, const uint16_t d, uint32_t (&v)[32]) {
        const __half2 d2 = __halves2half2(__ushort_as_half(d), __ushort_as_half(d));
        const uint32_t words[4] = {c.x, c.y, c.z, c.w};
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

// Sign bits: two 32-sign words per row and stage (bit b = element b of a
// word, set = +1); pair p = (element p, element p+16).  Activations staged in
// 32-element groups.  Raw stage: [128 rows][4 words], the words of stages
// kc & ~1 and kc | 1 (a TMA box is at least 16 bytes wide).
struct DecSign {
    static constexpr int RAW = UM_BM * 16;
    static constexpr bool DIRECT = false;
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
    __device__ __forceinline__ static void issue(const CUtensorMap* m0, const CUtensorMap*, uint8_t* raw,
                                                 uint64_t* bar, int row0, int kc) {
        tma_load_2d(raw, m0, bar, (kc >> 1) * 4, row0);        // x in words
    }
    __device__ __forceinline__ static void decode(const uint8_t* raw, int r, int kc, uint32_t (&v)[32]) {
        const uint2 w = *reinterpret_cast<const uint2*>(raw + r * 16 + (kc & 1) * 8);
        word(w.x, v);
        word(w.y, v + 16);
    }
    // a stage of KA = 2 or 4 atoms of 64 k: KA/2 boxes [128 rows][4 words]
    template <int KA>
    __host__ __device__ static constexpr int rawk() { return UM_BM * 8 * KA; }
    template <int KA>
    __device__ __forceinline__ static void issuek(const CUtensorMap* m0, const CUtensorMap*, uint8_t* raw,
                                                  uint64_t* bar, int row0, int ks) {
#pragma unroll
        for (int b = 0; b < KA / 2; ++b) tma_load_2d(raw + b * (UM_BM * 16), m0, bar, (ks * (KA / 2) + b) * 4, row0);
    }
    template <int KA>
    __device__ __forceinline__ static void decodek(const uint8_t* raw, int r, int p, uint32_t (&v)[32]) {
        decode(raw + (p >> 1) * (UM_BM * 16), r, p & 1, v);
    }
};

// Dense f16 rows, already in the K order the activations are staged in
// (pair j of a stage = elements 2j, 2j+1): TMA loads them as the A operand.
struct DecDense {
    static constexpr int RAW = 0;
    static constexpr bool DIRECT = true;
    __device__ __forceinline__ static void issue(const CUtensorMap* m0, const CUtensorMap*, uint8_t* a_stage,
                                                 uint64_t* bar, int row0, int kc) {
        tma_load_2d(a_stage, m0, bar, kc * UM_BK, row0);
    }
    __device__ __forceinline__ static void decode(const uint8_t*, int, int, uint32_t (&)[32]) {}
    template <int KA>
    __host__ __device__ static constexpr int rawk() { return 0; }   // one-atom stages only (the shared-memory A path)
};

// Host side: the tensor maps a plane's decoder loads from (PlaneMaps,
// tq2_internal.h).
// TQ2: stage-tiled codes [Rp/128][K/64][128][16 B] viewed as (128-byte line,
// line of the tile, tile); block-major scales [K/128][Rp] (Rp a multiple of 128)
inline bool plane_maps_tq2(PlaneMaps& pm, const uint8_t* codes_t, const uint16_t* scales_t, int K, int Rp) {
    const uint64_t dims[3] = {128u, (uint64_t)K / 4, (uint64_t)Rp / UM_BM};
    const uint64_t strides[2] = {128u, (uint64_t)K / 4 * 128u};
    const uint32_t box[3] = {128u, 16u, 1u};
    return make_tensor_map_3d(&pm.m0, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t*>(codes_t), dims, strides,
                              box, CU_TENSOR_MAP_SWIZZLE_NONE) &&
           make_tensor_map_2d(&pm.m1, CU_TENSOR_MAP_DATA_TYPE_UINT16, const_cast<uint16_t*>(scales_t), (uint64_t)Rp,
                              (uint64_t)K / 128, (uint64_t)Rp * 2, (uint32_t)UM_BM, 1u, CU_TENSOR_MAP_SWIZZLE_NONE);
}
// Sign: bits [R][K/32] u32 (K a multiple of 128)
inline bool plane_maps_sign(PlaneMaps& pm, const uint32_t* bits, int R, int K) {
    pm.m1 = CUtensorMap{};
    return make_tensor_map_2d(&pm.m0, CU_TENSOR_MAP_DATA_TYPE_UINT32, const_cast<uint32_t*>(bits), (uint64_t)K / 32,
                              (uint64_t)R, (uint64_t)K / 8, 4u, (uint32_t)UM_BM, CU_TENSOR_MAP_SWIZZLE_NONE);
}
// Dense: f16 rows [R][pitch] (pitch a multiple of 64)
inline bool plane_maps_dense(PlaneMaps& pm, const uint16_t* rows, int R, int pitch) {
    pm.m1 = CUtensorMap{};
    return make_tensor_map_2d(&pm.m0, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, const_cast<uint16_t*>(rows), (uint64_t)pitch,
                              (uint64_t)R, (uint64_t)pitch * 2, (uint32_t)UM_BK, (uint32_t)UM_BM,
                              CU_TENSOR_MAP_SWIZZLE_128B);
}

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
// activation tile in L2.  The stage rings and the two accumulators run
// continuously across tiles; the epilogue of a tile overlaps the MMAs of the
// next.
struct TileMap {
    // a unit is one weight tile x one token tile x one K split
    int tiles_n, tiles_np, tiles_m, splits, total, nk_total;
    __device__ __forceinline__ void decode(int t, int& np, int& m, int& z) const {
        np = t % tiles_np;
        const int rest = t / tiles_np;
        m = rest % tiles_m;
        z = rest / tiles_m;
    }
    // 32-bit arithmetic (nk_total * splits < 2^31): a 64-bit division is a
    // long software sequence on the GPU, paid on every tile by every role
    __device__ __forceinline__ int kc0(int z) const { return (nk_total * z) / splits; }
    __device__ __forceinline__ int kc1(int z) const { return (nk_total * (z + 1)) / splits; }
};

// AT: the decoded weights go to tensor memory (an S-stage ring of 32
// columns a stage after the NACC accumulators) instead of shared memory, and
// the MMAs read A from there; for token tiles of at most 128, where the
// shared-memory round trip of the decoded rows would cost more than the MMAs.
// KA > 1 (with AT): a pipeline stage spans KA x 64 k (KA 64-k swizzle atoms
// of activations, 32 KA tensor-memory columns of A, 4 KA MMAs), which cuts
// the per-stage waits, commits and hand-offs that set the pace of narrow
// token tiles; the MMA sequence, and so the result, is that of KA 64-k stages.
template <class Dec, int MODE, bool AT, int KA = 1>
__global__ void __launch_bounds__(UM_THREADS, 1)
umma_gemm_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap amap0,
                 const __grid_constant__ CUtensorMap amap1, const __grid_constant__ CUtensorMap omap,
                 const __grid_constant__ CUtensorMap imap, const EpiArgs ep, int T, int R, int BN, int tmem_cols,
                 const TileMap tm, int S, int SR, int NACC, int et) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int RAWB = KA > 1 ? Dec::template rawk<KA>() : Dec::RAW;   // raw plane bytes a stage
    const int stage_bytes = BN * 128 * KA;               // [KA][BN rows][128 B]
    uint8_t* a_ring = smem + S * stage_bytes;            // [S][128 rows][128 B], swizzled; 1 KB aligned (!AT)
    uint8_t* raw_ring = a_ring + (AT ? 0 : S * UM_A_STAGE);          // [SR][RAWB] (!DIRECT)
    UmmaBars* bars = reinterpret_cast<UmmaBars*>(raw_ring + (Dec::DIRECT ? 0 : SR * RAWB));
    // TMA epilogue (et): its input ring (column-sum modes) then the output
    // buffers (storing modes), 1 KB aligned after the barriers
    constexpr bool EPI_IN = MODE == EPI_COLSUM || MODE == EPI_SCALE_COLSUM;
    constexpr bool EPI_OUT = MODE != EPI_COLSUM;
    float* epi_in = reinterpret_cast<float*>(
        (reinterpret_cast<uintptr_t>(bars) + sizeof(UmmaBars) + 1023) & ~uintptr_t(1023));
    float* epi_out = epi_in + (EPI_IN ? UM_EPI_IN * UM_EPI_IN_BYTES / 4 : 0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit0 = blockIdx.x, units = gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < UM_STAGES; ++s) {
            mbar_init(&bars->full[s], Dec::DIRECT ? 1u : 5u);   // TMA producer (+ the stage's 4 decoder warps)
            mbar_init(&bars->empty[s], 1u);               // the MMA warp's commit releases it
        }
        for (int r = 0; r < UM_RAW_STAGES; ++r) {
            mbar_init(&bars->raw_full[r], 1);
            mbar_init(&bars->raw_empty[r], 4);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->acc_full[b], 1);
            mbar_init(&bars->acc_empty[b], 4);
        }
        for (int e = 0; e < UM_EPI_IN; ++e) {
            mbar_init(&bars->epi_full[e], 1);
            mbar_init(&bars->epi_empty[e], 4);
        }
        bars->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&xmap);
        tma_prefetch_desc(&amap0);
        if (!Dec::DIRECT) tma_prefetch_desc(&amap1);
        if (et && EPI_OUT) tma_prefetch_desc(&omap);
        if (et && EPI_IN) tma_prefetch_desc(&imap);
    }
    if (warp == 2) {
        tmem_alloc(&bars->tmem_base, (uint32_t)tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t a_col0 = (uint32_t)(NACC * BN);       // first column of the A ring (AT)
    constexpr uint32_t A_COLS = (uint32_t)(UM_BK / 2 * KA);   // tensor-memory columns of an A stage
    volatile int* abort_flag = &bars->abort;

    pdl_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {                                   // ---- activation TMA producer
            pdl_wait();
            int it = 0, s = 0;
            uint32_t ph = 0;                               // ring slot and phase parity of item `it`
            bool ok = true;
            const uint32_t tx = (uint32_t)stage_bytes + (Dec::DIRECT ? (uint32_t)UM_A_STAGE : 0u);
            for (int t = unit0; t < tm.total && ok && !*abort_flag; t += units) {
                int np, m, z;
                tm.decode(t, np, m, z);
                const int row0 = np * UM_BM;
                const int k1 = tm.kc1(z);
                for (int kc = tm.kc0(z); kc < k1; ++kc, ++it) {
                    if (it >= S && !mbar_wait_or_abort(&bars->empty[s], ph ^ 1u, abort_flag)) {
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars->full[s], tx);
                    // KA atoms of BN rows, each in boxes of at most 256 rows
                    // (the 384-token tile: three boxes of 128)
                    const int box = BN > UM_MAX_BN ? UM_BM : BN;
#pragma unroll
                    for (int a = 0; a < KA; ++a)
                        for (int r0 = 0; r0 < BN; r0 += box)
                            tma_load_2d(smem + s * stage_bytes + (a * BN + r0) * 128, &xmap, &bars->full[s],
                                        (kc * KA + a) * UM_BK, m * BN + r0);
                    if (Dec::DIRECT) Dec::issue(&amap0, &amap1, a_ring + s * UM_A_STAGE, &bars->full[s], row0, kc);
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
            }
            // let the copies already issued land before the CTA can exit
            for (int i = (it > S ? it - S : 0); i < it; ++i)
                mbar_wait(&bars->full[i % S], (uint32_t)(i / S) & 1u);
        }
    } else if (warp == 2) {
        if (EPI_IN && et && lane == 0) {                   // ---- TMA epilogue input producer
            // the column-sum operand, 32 tokens x 128 rows a chunk, in the
            // order the epilogue warps consume it
            pdl_wait();
            int c = 0, e = 0;
            uint32_t eph = 0;
            bool ok = true;
            for (int t = unit0; t < tm.total && ok && !*abort_flag; t += units) {
                int np, m, z;
                tm.decode(t, np, m, z);
                for (int cc = 0; cc < BN; cc += 32, ++c) {
                    if (c >= UM_EPI_IN && !mbar_wait_or_abort(&bars->epi_empty[e], eph ^ 1u, abort_flag)) {
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars->epi_full[e], (uint32_t)UM_EPI_IN_BYTES);
                    tma_load_2d(epi_in + e * (UM_EPI_IN_BYTES / 4), &imap, &bars->epi_full[e], np * UM_BM,
                                m * BN + cc);
                    if (++e == UM_EPI_IN) { e = 0; eph ^= 1u; }
                }
            }
            for (int i = (c > UM_EPI_IN ? c - UM_EPI_IN : 0); i < c; ++i)
                mbar_wait(&bars->epi_full[i % UM_EPI_IN], (uint32_t)(i / UM_EPI_IN) & 1u);
        }
    } else if (warp == 3) {
        if (!Dec::DIRECT && lane == 0) {                   // ---- plane TMA producer (raw stages)
            pdl_wait();
            int it = 0, r = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int t = unit0; t < tm.total && ok && !*abort_flag; t += units) {
                int np, m, z;
                tm.decode(t, np, m, z);
                const int row0 = np * UM_BM;
                const int k1 = tm.kc1(z);
                for (int kc = tm.kc0(z); kc < k1; ++kc, ++it) {
                    if (it >= SR && !mbar_wait_or_abort(&bars->raw_empty[r], ph ^ 1u, abort_flag)) {
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars->raw_full[r], (uint32_t)RAWB);
                    if constexpr (KA > 1)
                        Dec::template issuek<KA>(&amap0, &amap1, raw_ring + r * RAWB, &bars->raw_full[r], row0, kc);
                    else
                        Dec::issue(&amap0, &amap1, raw_ring + r * RAWB, &bars->raw_full[r], row0, kc);
                    if (++r == SR) { r = 0; ph ^= 1u; }
                }
            }
            for (int i = (it > SR ? it - SR : 0); i < it; ++i)
                mbar_wait(&bars->raw_full[i % SR], (uint32_t)(i / SR) & 1u);
        }
    } else if (warp == 1) {
        // ---- MMA issuer.  The tensor pipe holds about one MMA beyond the one
        // executing, so whatever this warp does between two stages idles it:
        // the whole warp waits (no lane-0 wait and broadcast), a stage has one
        // barrier (B bytes and decoded A together), and the next stage's
        // barrier is tested without blocking before this stage's MMAs are
        // issued, so a stage that is already complete costs no wait at all.
        // Every MMA and commit is issued by one lane chosen with elect.sync.
        const uint32_t idesc = idesc_f16_f32(UM_BM, (uint32_t)(BN > UM_MAX_BN ? UM_MAX_BN : BN));
        const uint32_t idesc2 = idesc_f16_f32(UM_BM, (uint32_t)(BN > UM_MAX_BN ? BN - UM_MAX_BN : 16));
        int lt = 0, s = 0;
        uint32_t ph = 0;
        bool ok = true;
        bool ready = false;                                // full[s] of the next stage known complete
        auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {   // warp-uniform result
            return __all_sync(0xffffffffu, mbar_wait_or_abort(bar, parity, abort_flag, true)) != 0;
        };
        for (int t = unit0; t < tm.total && ok; t += units, ++lt) {
            int np, m, z;
            tm.decode(t, np, m, z);
            const int buf = NACC == 2 ? (lt & 1) : 0, use = NACC == 2 ? (lt >> 1) : lt;
            if (use >= 1 && !wait_all(&bars->acc_empty[buf], (uint32_t)(use - 1) & 1u)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const uint32_t dcol = tmem + (uint32_t)(buf * BN);
            const int k0 = tm.kc0(z), k1 = tm.kc1(z);
            for (int kc = k0; kc < k1; ++kc) {
                if (!ready && !wait_all(&bars->full[s], ph)) {
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                const int s1 = s + 1 == S ? 0 : s + 1;
                const uint32_t ph1 = s + 1 == S ? ph ^ 1u : ph;
                ready = mbar_test_wait(&bars->full[s1], ph1);   // its latency hides under the MMAs below
                tc_fence_after();
                const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(smem + s * stage_bytes));
                if (AT && KA > 1) {
                    // atom a of the B stage at a * BN rows; k-step j of atom a at A column (4a + j) * 8
                    const uint32_t acol = tmem + a_col0 + (uint32_t)s * A_COLS;
#pragma unroll
                    for (int a = 0; a < KA; ++a) {
                        const uint64_t bda = sdesc_kmajor_sw128(smem_u32(smem + s * stage_bytes + a * BN * 128));
#pragma unroll
                        for (int j = 0; j < UM_BK / 16; ++j)
                            umma_f16_ts_elect(dcol, acol + (uint32_t)((a * (UM_BK / 16) + j) * 8),
                                              bda + (uint64_t)(2 * j), idesc, (kc > k0 || a > 0 || j > 0) ? 1u : 0u);
                    }
                } else if (AT) {
                    const uint32_t acol = tmem + a_col0 + (uint32_t)(s * (UM_BK / 2));
                    if (BN > UM_MAX_BN) {
                        // tokens 256.. of the tile: rows 256.. of the B stage (1 KB swizzle atoms)
                        const uint64_t bdesc2 = sdesc_kmajor_sw128(smem_u32(smem + s * stage_bytes + UM_MAX_BN * 128));
#pragma unroll
                        for (int j = 0; j < UM_BK / 16; ++j) {
                            const uint32_t acc = (kc > k0 || j > 0) ? 1u : 0u;
                            umma_f16_ts_elect(dcol, acol + (uint32_t)(j * 8), bdesc + (uint64_t)(2 * j), idesc, acc);
                            umma_f16_ts_elect(dcol + (uint32_t)UM_MAX_BN, acol + (uint32_t)(j * 8),
                                              bdesc2 + (uint64_t)(2 * j), idesc2, acc);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < UM_BK / 16; ++j)
                            umma_f16_ts_elect(dcol, acol + (uint32_t)(j * 8), bdesc + (uint64_t)(2 * j), idesc,
                                              (kc > k0 || j > 0) ? 1u : 0u);
                    }
                } else {
                    const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(a_ring + s * UM_A_STAGE));
#pragma unroll
                    for (int j = 0; j < UM_BK / 16; ++j)
                        umma_f16_ss_elect(dcol, adesc + (uint64_t)(2 * j), bdesc + (uint64_t)(2 * j), idesc,
                                          (kc > k0 || j > 0) ? 1u : 0u);
                }
                umma_commit_elect(&bars->empty[s]);
                s = s1;
                ph = ph1;
                ready = __all_sync(0xffffffffu, ready);
            }
            if (!ok) break;
            umma_commit_elect(&bars->acc_full[buf]);
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        }
    } else if (warp >= 4 && warp < 12) {                   // ---- decoders
        if (!Dec::DIRECT) {
            // warp pair (q, h): lane quarter q, the items (stages) of parity h
            // of the CTA's item sequence; the loop visits only those.  A
            // stage's raw tile is in shared memory (it landed S_R stages ahead).
            const int q = warp & 3, h = (warp - 4) >> 2;
            const int arow = q * 32 + lane;                // row of the tile this thread decodes
            int it = 0, s = 0, r = 0;
            uint32_t ph = 0, rph = 0;                      // A-ring and raw-ring phase parities of item `it`
            auto advance = [&](int n) {                    // n <= 2 <= S, SR
                it += n;
                s += n;
                if (s >= S) { s -= S; ph ^= 1u; }
                r += n;
                if (r >= SR) { r -= SR; rph ^= 1u; }
            };
            if (h) advance(1);
            int lead = h;                                  // first own item's offset into the next tile
            bool ok = true;
            for (int t = unit0; t < tm.total && ok; t += units) {
                int np, m, z;
                tm.decode(t, np, m, z);
                const int k1 = tm.kc1(z);
                int kc = tm.kc0(z) + lead;
                for (; kc < k1; kc += 2, advance(2)) {
                    if (!mbar_wait_or_abort(&bars->raw_full[r], rph, abort_flag)) {
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    uint32_t v[32];
                    if constexpr (KA > 1) {
                        // multi-atom stage: each 64-k atom decoded and stored in
                        // turn (one 32-register array; its store completes
                        // before the array is reused)
                        if (it >= S && !mbar_wait_or_abort(&bars->empty[s], ph ^ 1u, abort_flag)) {
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t acol = tmem + ((uint32_t)(q * 32) << 16) + a_col0 + (uint32_t)s * A_COLS;
#pragma unroll
                        for (int p = 0; p < KA; ++p) {
                            Dec::template decodek<KA>(raw_ring + r * RAWB, arow, p, v);
                            if (p == KA - 1) {
                                fence_proxy_async_shared();    // raw reads done: the slot is refilled
                                __syncwarp();                  // through the async proxy
                                if (lane == 0) mbar_arrive(&bars->raw_empty[r]);
                            }
                            tmem_st_32x32b_x32(acol + (uint32_t)(p * (UM_BK / 2)), v);
                            tmem_wait_st();
                        }
                        tc_fence_before();
                    } else {
                        Dec::decode(raw_ring + r * RAWB, arow, kc, v);
                        // the raw slot is refilled through the async proxy
                        fence_proxy_async_shared();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars->raw_empty[r]);
                        if (it >= S && !mbar_wait_or_abort(&bars->empty[s], ph ^ 1u, abort_flag)) {
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        if (AT) {
                            // row arow = TMEM lane arow; pair j of the stage in column j of the stage's 32
                            tc_fence_after();
                            tmem_st_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + a_col0 + (uint32_t)(s * (UM_BK / 2)),
                                               v);
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
                            fence_proxy_async_shared();    // the MMA reads A through the async proxy
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->full[s]);
                }
                lead = kc - k1;                            // 0, or 1 when the tile's last item was not ours
            }
        }
    } else if (warp >= 12) {                               // ---- epilogue
        const int q = warp & 3;
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        bool waited = false;
        int lt = 0;
        int ec = 0, e = 0, ob = 0;                         // TMA epilogue: chunk count, input slot, output buffer
        uint32_t eph = 0;
        for (int t = unit0; t < tm.total; t += units, ++lt) {
            int np, m, z;
            tm.decode(t, np, m, z);
            const int n = np;
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
            if (et) {
                // 32 tokens at a time: the column-sum operand from the input
                // ring (this warp's 32 rows of the chunk), the results through
                // a [32 tokens][32 rows] buffer and one TMA store (tokens past
                // T and rows past R are neither read nor written)
                bool fail = false;
                for (int cc = 0; cc < BN; cc += 32, ++ec) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(lane_addr + (uint32_t)(buf * BN + cc), v);
                    tmem_wait_ld();
                    if (cc + 32 >= BN) {                   // accumulator fully read: hand it back
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars->acc_empty[buf]);
                    }
                    const float* in = epi_in + e * (UM_EPI_IN_BYTES / 4) + q * 32 + lane;   // token i at in[128 i]
                    float* o = epi_out + (q * 2 + ob) * 1024;                              // token i at o[32 i + lane]
                    if (EPI_IN && !mbar_wait_or_abort(&bars->epi_full[e], eph, abort_flag)) {
                        *abort_flag = 1;
                        fail = true;
                        break;
                    }
                    if (EPI_OUT) {
                        if (lane == 0) bulk_wait_group_read<1>();   // this buffer's store (two chunks back) has read it
                        __syncwarp();
                    }
                    // columns past the accumulator (a tile narrower than a
                    // multiple of 32) hold other data: stored only where the
                    // TMA clips them (tokens past T), and kept out of the sums
                    const int nvalid = (T - (m0 + cc)) < 32 ? (T - (m0 + cc)) : 32;
                    auto one = [&](int i, bool valid) {
                        const float w = __uint_as_float(v[i]) * ep.oscale;
                        if (MODE == EPI_STORE) o[32 * i + lane] = w;
                        if (MODE == EPI_SCALE || MODE == EPI_SCALE_COLSUM) o[32 * i + lane] = __fmul_rn(w, vs);
                        if (EPI_IN && valid) colacc = fmaf(w, in[128 * i], colacc);
                    };
                    if (nvalid == 32) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) one(i, true);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) one(i, i < nvalid);
                    }
                    if (EPI_IN) {
                        fence_proxy_async_shared();        // the slot is refilled through the async proxy
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars->epi_empty[e]);
                        if (++e == UM_EPI_IN) { e = 0; eph ^= 1u; }
                    }
                    if (EPI_OUT) {
                        fence_proxy_async_shared();        // the TMA store reads the buffer through the async proxy
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&omap, o, n * UM_BM + q * 32, m0 + cc);
                            bulk_commit_group();
                        }
                        ob ^= 1;
                    }
                }
                if (fail) break;
                if ((MODE == EPI_SCALE_COLSUM || MODE == EPI_COLSUM) && rok)
                    ep.colpart[(int64_t)m * ep.ldo + row] = colacc;
                continue;
            }
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
                // both paths fully unrolled (a runtime index into v would put it
                // in local memory); the full one without predicates
                if (nvalid == 32) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) one(i);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i < nvalid) one(i);
                }
            }
            if ((MODE == EPI_SCALE_COLSUM || MODE == EPI_COLSUM) && rok)
                ep.colpart[(int64_t)m * ep.ldo + row] = colacc;
        }
        if (et && EPI_OUT && lane == 0) bulk_wait_group<0>();   // this warp's stores are complete
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)tmem_cols);
    }
}

// Host: launch one GEMM.  act16 is f16 [T][K] (row pitch K), staged in the
// decoder's K order; R = plane rows; splits = K splits; pm = the plane's
// tensor maps.  Token tiles of at most 128, the ternary GEMM's 256-token
// tiles and the 384-token wide tile keep the decoded weights in tensor memory
// (AT); the blr GEMMs' 256-token tiles decode into shared memory, and dense
// planes always take the shared-memory path (TMA writes A).  Every CTA loads
// its own activation tile: pairs of CTAs sharing it measured slower at 256
// tokens and the same for the wide tile.
template <class Dec, int MODE, bool AT, int KA>
cudaError_t launch_umma_impl(const PlaneMaps& pm, const EpiArgs& ep, const void* act16, int T, int R, int K, int BN,
                             int splits, cudaStream_t st) {
    const bool wide = BN == UM_WIDE_BN;
    if ((BN > UM_MAX_BN && !wide) || BN % 16 != 0 || BN < 16 || (AT && BN > 128 && !wide && BN != UM_MAX_BN) || (wide && !AT))
        return cudaErrorInvalidValue;
    // multi-atom stages: tensor-memory A, every K split at least one stage
    if (KA > 1 && (!AT || wide || Dec::DIRECT || K % (UM_BK * KA) != 0 || splits > K / (UM_BK * KA)))
        return cudaErrorInvalidValue;
    // the epilogue drains 32 columns at a time: a tile narrower than a
    // multiple of 32 must be the only token tile
    if (BN % 32 != 0 && T > BN) return cudaErrorInvalidValue;
    const int tiles_n = (R + UM_BM - 1) / UM_BM;
    CUtensorMap xmap;                                     // a TMA box is at most 256 rows
    if (!make_tensor_map_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, const_cast<void*>(act16), (uint64_t)K,
                            (uint64_t)T, (uint64_t)K * 2, UM_BK, (uint32_t)(BN > UM_MAX_BN ? UM_BM : BN),
                            CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    // two accumulators in tensor memory (the epilogue of a tile overlaps the
    // next tile's MMAs), one for the wide tile (its epilogue, ~3 % of a
    // tile's K loop, stalls the MMAs); the B ring (and the A ring unless AT)
    // in shared memory, then the raw plane ring with what is left; with AT
    // the A ring takes S x 32 tensor-memory columns after the accumulators
    // (2 x 128 + 8 x 32 or 384 + 4 x 32 = 512 at most)
    const int NACC = (wide || (AT && BN > 128)) ? 1 : 2;   // one accumulator when A takes its room
    const int a_stage = AT ? 0 : UM_A_STAGE;
    const int raw = Dec::DIRECT ? 0 : (KA > 1 ? Dec::template rawk<KA>() : Dec::RAW);
    const int b_stage = BN * 128 * KA;
    const int a_cols = UM_BK / 2 * KA;                    // tensor-memory columns of an A stage (AT)
    // TMA epilogue (et) for the column-sum modes (without accumulation into
    // the output) of GEMMs of at most UM_EPI_TMA_STEPS 64-k steps a tile,
    // whose epilogue is not hidden behind the next tile's MMAs; needs 16-byte
    // rows and bases, no K split.  (Plain and scaled stores
    // through it measured slower: the blr forward 41.8 -> 42.8 us.)
    constexpr bool EPI_IN = MODE == EPI_COLSUM || MODE == EPI_SCALE_COLSUM;
    constexpr bool EPI_OUT = MODE != EPI_COLSUM;
    const bool epi_mode = MODE == EPI_COLSUM || (MODE == EPI_SCALE_COLSUM && !ep.accumulate);
    const bool epi_aligned = ep.ldo % 4 == 0 && (!EPI_OUT || (reinterpret_cast<uintptr_t>(ep.out) & 15) == 0) &&
                             (!EPI_IN || (reinterpret_cast<uintptr_t>(ep.other) & 15) == 0);
    int et = (epi_mode && epi_aligned && splits == 1 && K / UM_BK <= UM_EPI_TMA_STEPS) ? 1 : 0;
    int S = 0, SR = 0;
    size_t epi_bytes = 0;
    for (;; et = 0) {
        epi_bytes = et ? (size_t)(EPI_IN ? UM_EPI_IN * UM_EPI_IN_BYTES : 0) + (EPI_OUT ? UM_EPI_OUT_BYTES : 0) + 1024
                       : 0;
        const size_t budget = (size_t)220 * 1024 - sizeof(UmmaBars) - 1024 - epi_bytes;
        S = UM_STAGES;
        if (AT && S > (512 - NACC * BN) / a_cols) S = (512 - NACC * BN) / a_cols;   // A ring in tensor memory
        // leave room for at least 8 raw stages (4 beside the TMA epilogue's
        // buffers, where a third stage measured faster than four more raw
        // slots: the blr backward 72 -> 70 us)
        while (S > 2 && (size_t)S * (b_stage + a_stage) + (size_t)(et || (AT && BN > 128) ? 4 : 8) * raw > budget)
            --S;
        SR = 0;
        if ((size_t)S * (b_stage + a_stage) < budget)
            SR = Dec::DIRECT ? 2 : (int)((budget - (size_t)S * (b_stage + a_stage)) / (size_t)(raw > 0 ? raw : 1));
        if (SR > UM_RAW_STAGES) SR = UM_RAW_STAGES;
        // an even depth: the two decoder warps of a quarter take alternate items,
        // so items it and it + SR (one raw slot) belong to the same warp and no
        // warp can wait on a slot's phase a ring round ahead of its filling
        SR &= ~1;
        if ((S >= 2 && SR >= 2) || !et) break;
    }
    if (S < 2 || SR < 2) return cudaErrorInvalidValue;
    CUtensorMap omap{}, imap{};
    if (et && EPI_OUT &&
        !make_tensor_map_2d(&omap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ep.out, (uint64_t)ep.ldo, (uint64_t)T,
                            (uint64_t)ep.ldo * 4, 32u, 32u, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    if (et && EPI_IN &&
        !make_tensor_map_2d(&imap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, const_cast<float*>(ep.other), (uint64_t)ep.ldo,
                            (uint64_t)T, (uint64_t)ep.ldo * 4, (uint32_t)UM_BM, 32u, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    int tmem_cols = 32;
    while (tmem_cols < NACC * BN + (AT ? S * a_cols : 0)) tmem_cols <<= 1;
    if (tmem_cols > 512) return cudaErrorInvalidValue;
    // At least 120 KB of shared memory: no two CTAs of this kernel can share
    // an SM, so a CTA never waits in tcgen05.alloc for a co-resident CTA.
    size_t smem = (size_t)S * (b_stage + a_stage) + (Dec::DIRECT ? 0 : (size_t)SR * raw) + 1024 + sizeof(UmmaBars) +
                  1024 + epi_bytes;
    if (smem < (size_t)120 * 1024) smem = (size_t)120 * 1024;
    TileMap tm;
    tm.tiles_n = tiles_n;
    tm.tiles_np = tiles_n;
    tm.tiles_m = (T + BN - 1) / BN;
    tm.splits = splits;
    tm.total = tm.tiles_np * tm.tiles_m * splits;
    tm.nk_total = K / (UM_BK * KA);
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int units = tm.total < sms ? tm.total : sms;
    cudaError_t e = cudaFuncSetAttribute(umma_gemm_kernel<Dec, MODE, AT, KA>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)units);
    cfg.blockDim = dim3(UM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, umma_gemm_kernel<Dec, MODE, AT, KA>, xmap, pm.m0, pm.m1, omap, imap, ep, T, R, BN,
                              tmem_cols, tm, S, SR, NACC, et);
}

template <class Dec, int MODE>
cudaError_t launch_umma(const PlaneMaps& pm, const EpiArgs& ep, const void* act16, int T, int R, int K, int BN,
                        int splits, cudaStream_t st) {
    if constexpr (!Dec::DIRECT) {
        // token tiles of at most 128: stages of 256 k (tensor memory holds
        // two to three of them after the accumulators: at 32 tokens 19.6 ->
        // 16.6 us and at 128 tokens 20.5 -> 19.6 us against 128-k stages, at
        // N=11008, K=4096), else 128 k, when every K split keeps at least one
        if (BN <= 128 && K % (4 * UM_BK) == 0 && splits <= K / (4 * UM_BK))
            return launch_umma_impl<Dec, MODE, true, 4>(pm, ep, act16, T, R, K, BN, splits, st);
        if (BN <= 128 && K % (2 * UM_BK) == 0 && splits <= K / (2 * UM_BK))
            return launch_umma_impl<Dec, MODE, true, 2>(pm, ep, act16, T, R, K, BN, splits, st);
        if (BN <= 128 || BN == UM_WIDE_BN)
            return launch_umma_impl<Dec, MODE, true, 1>(pm, ep, act16, T, R, K, BN, splits, st);
        // 256 tokens, plain or split-K stores (the ternary GEMM): A in tensor
        // memory too, in 128-k stages, with one 256-column accumulator (the
        // tile's epilogue then holds the MMAs, a few % of a tile) and three
        // 64 KB activation stages: M=4096 x N=14336 302 -> 287 us, DiT
        // N=3072 29.5 -> 28.3 us.  The column-sum modes keep the
        // shared-memory A path and its room for the TMA epilogue.
        if ((MODE == EPI_STORE || MODE == EPI_ATOMIC) && BN == UM_MAX_BN && K % (2 * UM_BK) == 0 &&
            splits <= K / (2 * UM_BK))
            return launch_umma_impl<Dec, MODE, true, 2>(pm, ep, act16, T, R, K, BN, splits, st);
    }
    return launch_umma_impl<Dec, MODE, false, 1>(pm, ep, act16, T, R, K, BN, splits, st);
}

inline int umma_pick_bn(int T) {
    if (T >= 256) return 256;
    return ((T + 15) / 16) * 16;
}

}  // namespace tq2
