// tq2_gemv.cu -- fused decode-shape GEMV for M <= 8 tokens.
//
//   out[m,n] = sum_k x[m,k] * W[n,k],  W[n,k] = (c-1)*d   (BlockTQ2_0_g128,
//   "oxibonsai-kernels 0.2.1, src/gpu_backend/metal_graph/tests_gemm_tq2.rs")
//
// One kernel per launch (one GEMV, or up to 64 independent GEMVs sharing K and
// M), no scratch.  A CTA is one producer warp and eight consumer warps; it
// owns a contiguous range of work units.
//
//   * The producer streams the weights.  A stage is 16 KB of codes fetched by
//     ONE TMA load through a 3D view of the code plane -- (128-byte piece,
//     row, piece index) -- with 128-byte swizzling, so each warp's share
//     lands as [16 rows][128 B] (4 blocks of 128 k per row) and the MMA
//     fragments read back without bank conflicts.  Per unit one
//     cp.async.bulk brings the unit's block scales (consecutive rows' scales
//     are contiguous in the scale plane) into a ring of slots.  The weights
//     never depend on earlier work on the stream, so this starts at once.
//   * The consumers wait for the previous kernel (griddepcontrol.wait),
//     convert x once into the hi/lo f16 B fragments of mma.m16n8k16 in
//     shared memory (B column 2m = token m's hi part, 2m+1 its lo part; M
//     is padded to MT in {1, 2, 4, 8} tokens, so one n8 tile holds up to four
//     tokens and MT = 8 takes two), then per stage decode their 4 blocks
//     (shift + mask|magic, see gv_pair) and issue the MMAs -- each decoded
//     A fragment feeds every n8 tile: one accumulator chain per block and
//     tile, the blocks' chains interleaved per warp, f32 accumulate, block
//     scale applied to the block result d * (acc - correction).  The correction
//     sum_k (m_q+1) x_k of a block is computed by the very MMA chain that a
//     block of all code-1 weights takes, so such a block gives exactly 0 and
//     the rounding error of a block scales with its nonzero weights.
//   * Two ways to cut the work (the smem addressing of a warp's share is the
//     same in both):
//       k-split (small N): a unit is 16 rows; a stage covers them over 32
//         blocks, warp w taking blocks 4w..4w+3; the warps' sums meet in
//         shared memory and are added in a fixed order.
//       row-split (N large enough to fill the GPU): a unit is 128 rows; a
//         stage covers them over 4 blocks, warp w taking rows 16w..16w+15
//         over all of K, so no cross-warp reduction is needed.  Each warp
//         keeps eight partial sums that mirror the k-split warps, so both
//         ways give bit-identical results.
// Row-split launches keep shared memory under ~110 KB so that two CTAs share
// an SM; k-split launches run one CTA on every SM, under ~110 KB where x
// leaves room for four stages, so the next kernel on the stream (launched
// early through programmatic dependent launch) fits beside it and streams
// its own weights.
#include "ptx.cuh"
#include "tq2_internal.h"

namespace tq2 {

namespace {

constexpr int GV_CONS = 8;                         // consumer warps
constexpr int GV_THREADS = (GV_CONS + 1) * 32;     // + one producer warp
constexpr int GV_BPW = 4;                          // 128-blocks per consumer warp per stage
constexpr int GV_PIECE = 128;                      // bytes of one row's codes for 4 blocks
constexpr int GV_WARP_BYTES = 16 * GV_PIECE;       // a warp's share of a stage: 16 rows x 128 B
constexpr int GV_STAGE = GV_CONS * GV_WARP_BYTES;  // 16 KB
constexpr int GV_MAX_STAGES = 16;
constexpr int GV_MAX_SSLOTS = 8;                   // scale slots (one unit each)
constexpr int GV_SMEM_PAIR = 110 * 1024;           // two CTAs per SM (with the static job table)
constexpr int GV_SMEM_MAX = 225 * 1024;            // dynamic part; + up to 2 KB static job table

enum GvMode { GV_KSPLIT = 0, GV_ROWS = 1 };
__host__ __device__ constexpr int gv_unit_rows(int mode) { return mode == GV_ROWS ? 16 * GV_CONS : 16; }
__host__ __device__ constexpr int gv_stage_blocks(int mode) { return mode == GV_ROWS ? GV_BPW : GV_BPW * GV_CONS; }
// tokens padded to MT in {1, 2, 4, 8}; B columns 2MT in one or two n8 tiles
__host__ __device__ constexpr int gv_mt(int M) { return M <= 2 ? M : (M <= 4 ? 4 : 8); }
__host__ __device__ constexpr int gv_tiles(int MT) { return MT > 4 ? 2 : 1; }

struct GemvJob {
    CUtensorMap map;              // the weight's code-plane map for the launch's mode
    const uint16_t* scales;
    const float* x;
    float* out;
    int N;
    int unit0;                    // first unit of this job in the launch
};
template <int NJ>
struct GemvTab {
    GemvJob job[NJ];
    int njobs;
    int K;
    int M;                        // tokens (<= MT; the rest of the MT columns are zero)
};

// The per-job fields the loops read, copied to shared memory once: the job
// table is a kernel parameter, and reading it with a runtime index goes
// through the constant cache.
struct GvJobS {
    const uint16_t* scales;
    const float* x;
    float* out;
    int N, unit0;
};

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);      // .x (low 16 bits) = lo
    return *reinterpret_cast<const uint32_t*>(&h);
}

// hi = f16(v), lo = f16(v - hi): the pair as two f16x2 words.
__device__ __forceinline__ void split2(float v0, float v1, uint32_t& hi, uint32_t& lo) {
    const __half2 h = __floats2half2_rn(v0, v1);
    const float2 back = __half22float2(h);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = pack_h2(v0 - back.x, v1 - back.y);
}

// Pair q of a 16-code word (elements q and q+8 at bits 2q and 16+2q) as the
// exact f16 pair (m_q + c_lo, m_q + c_hi): the code is brought to bit
// P in {4, 6, 8} of each half by one of two shifts (or none) and OR-ed into
// the mantissa of m_q = 2^(10-P).
//   q:    0   1   2   3   4   5   6   7
//   word: <<4 <<4  .   .   .  >>6 >>6 >>6
//   P:    4   6   4   6   8   4   6   8
//   m_q:  64  16  64  16  4   64  16  4
// The integer ALU pipe runs at half rate and is the decode's bottleneck, so:
//   * the two shifts are integer multiplies (w * 16, and the high half of
//     w * 2^26) by factors the compiler cannot fold, which run on the FMA pipe;
//   * the three masks sit in registers, so (w & mask) | magic is a single
//     three-input logic op with the magic as its one immediate.
struct GvShift {
    uint32_t m16, m2p26;         // 16 and 2^26
    uint32_t k4, k6, k8;         // 0x00030003 << 4, << 6, << 8
};
template <int P>
__device__ __forceinline__ uint32_t gv_op(uint32_t ws, uint32_t mask) {
    constexpr uint32_t mh = (uint32_t)(25 - P) << 10;     // f16 bits of 2^(10-P)
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(ws), "r"(mask), "n"(mh | (mh << 16)));   // (a & b) | c
    return r;
}
template <int Q>
__device__ __forceinline__ uint32_t gv_pair(uint32_t w, uint32_t wl, uint32_t wr, const GvShift& sh) {
    if constexpr (Q == 0) return gv_op<4>(wl, sh.k4);
    else if constexpr (Q == 1) return gv_op<6>(wl, sh.k6);
    else if constexpr (Q == 2) return gv_op<4>(w, sh.k4);
    else if constexpr (Q == 3) return gv_op<6>(w, sh.k6);
    else if constexpr (Q == 4) return gv_op<8>(w, sh.k8);
    else if constexpr (Q == 5) return gv_op<4>(wr, sh.k4);
    else if constexpr (Q == 6) return gv_op<6>(wr, sh.k6);
    else return gv_op<8>(wr, sh.k8);
}
// The A fragment of k16 step j (0..3) of a word: rows g and g+8 from words
// wa and wb; positions 2t,2t+1 hold pair 2j, positions 2t+8,2t+9 pair 2j+1.
template <int J>
__device__ __forceinline__ void gv_afrag(const uint32_t (&wa)[3], const uint32_t (&wb)[3], uint32_t (&a)[4],
                                         const GvShift& sh) {
    a[0] = gv_pair<2 * J>(wa[0], wa[1], wa[2], sh);
    a[1] = gv_pair<2 * J>(wb[0], wb[1], wb[2], sh);
    a[2] = gv_pair<2 * J + 1>(wa[0], wa[1], wa[2], sh);
    a[3] = gv_pair<2 * J + 1>(wb[0], wb[1], wb[2], sh);
}
// A word with its two shifted copies: w, w << 4, w >> 6.
__device__ __forceinline__ void gv_word(uint32_t w, const GvShift& sh, uint32_t (&o)[3]) {
    o[0] = w;
    o[1] = w * sh.m16;
    o[2] = __umulhi(w, sh.m2p26);
}

struct GvLayout {
    int nb, nch;
    uint32_t off_red, off_corr, off_sc, sc_bytes, off_xs, off_ring, total;
};

// Shared-memory carve (byte offsets from the dynamic base; barriers first).
__host__ __device__ inline GvLayout gv_layout(int K, int MT, int mode, int stages, int sslots) {
    GvLayout L;
    L.nb = K / 128;
    L.nch = (L.nb + gv_stage_blocks(mode) - 1) / gv_stage_blocks(mode);
    L.off_red = 512;                                                   // full, empty, sfull, sempty
    L.off_corr = L.off_red + (mode == GV_KSPLIT ? 2u * GV_CONS * 16 * MT * 4 : 0u);
    L.off_sc = L.off_corr + (((uint32_t)L.nb + 3u) & ~3u) * MT * 4;             // [MT][nb rounded to 4] (float4 reads)
    L.sc_bytes = ((uint32_t)gv_unit_rows(mode) * L.nb * 2 + 16u + 15u) & ~15u;
    L.off_xs = L.off_sc + (uint32_t)sslots * L.sc_bytes;
    // [nb rounded up to whole pieces][4 step pairs][2MT][4] uint4
    L.off_ring = L.off_xs + (((uint32_t)L.nb + 3u) & ~3u) * 4 * (2 * MT) * 4 * 16;
    L.total = L.off_ring + 1024u + (uint32_t)stages * GV_STAGE;                  // + room to align to 1 KB
    return L;
}

// One warp's share of a stage: 4 consecutive blocks blk0.. of rows g and g+8
// (nv of them valid).  pc points at the warp's 2 KB region + g*128 + 8*(t&1);
// 16-byte chunk (2i + t/2) of a 128-byte row is stored at chunk
// (2i + t/2) ^ (row & 7), and row g+8 sits 1 KB after row g.  scA points at
// row g's scales (row g+8's are 8*nb further).  x fragments are stored
// [block][k16 step pair][column][t] (uint4 = two steps' b0,b1), so the
// lanes of one load read 16 * 8 * MT contiguous bytes; xl is this lane's
// fragment base in n8 tile 0 (tile 1, columns 8..15, is 32 uint4 further),
// xstep / sstep its strides per block / step pair.  Lanes g >= 2MT supply B
// columns whose D columns are never read, so they load another lane's
// fragment (a broadcast).  cr points at the corrections of this lane's
// token of tile 0 (tile 1's token, 4 later, is 4*nbp further).  Each block
// and tile's eight MMAs form one accumulator chain; the chains interleave.
template <int MT, bool FULL>
__device__ __forceinline__ void gv_piece(const uint8_t* pc, int g, int t, const uint4* xl, int xstep, int sstep,
                                         const float* cr, int nbp, int blk0, int nv, int nb, const uint16_t* scA,
                                         const GvShift& sh, float (&totA)[gv_tiles(MT)], float (&totB)[gv_tiles(MT)]) {
    constexpr int NT = gv_tiles(MT);
    uint32_t wa[GV_BPW][2][3], wb[GV_BPW][2][3];
    const uint4* xb = xl + blk0 * xstep;
#pragma unroll
    for (int i = 0; i < GV_BPW; ++i) {
        const uint8_t* p = pc + ((((2 * i + (t >> 1)) ^ g) & 7) << 4);
        const uint2 ca = *reinterpret_cast<const uint2*>(p);
        const uint2 cb = *reinterpret_cast<const uint2*>(p + 8 * GV_PIECE);
        gv_word(ca.x, sh, wa[i][0]);
        gv_word(ca.y, sh, wa[i][1]);
        gv_word(cb.x, sh, wb[i][0]);
        gv_word(cb.y, sh, wb[i][1]);
    }
    float acc[GV_BPW][NT][4];
#pragma unroll
    for (int i = 0; i < GV_BPW; ++i)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[i][j][q] = 0.f;
    // steps 0-3 decode word x (k 32t..32t+15 of the block), 4-7 word y
#define GV_STEP2(S)                                                                         \
    _Pragma("unroll") for (int i = 0; i < GV_BPW; ++i) {                                    \
        uint4 b[NT];                                                                        \
        _Pragma("unroll") for (int j = 0; j < NT; ++j) b[j] = xb[i * xstep + ((S) / 2) * sstep + 32 * j]; \
        uint32_t a[4];                                                                      \
        gv_afrag<(S) % 4>(wa[i][(S) / 4], wb[i][(S) / 4], a, sh);                           \
        _Pragma("unroll") for (int j = 0; j < NT; ++j) mma_16816_pure(acc[i][j], a, b[j].x, b[j].y); \
        gv_afrag<((S) + 1) % 4>(wa[i][(S) / 4], wb[i][(S) / 4], a, sh);                     \
        _Pragma("unroll") for (int j = 0; j < NT; ++j) mma_16816_pure(acc[i][j], a, b[j].z, b[j].w); \
    }
    GV_STEP2(0)
    GV_STEP2(2)
    GV_STEP2(4)
    GV_STEP2(6)
#undef GV_STEP2
    // block scales (f16) and corrections of the four blocks
    float dA[GV_BPW], dB[GV_BPW];
    if ((nb & 3) == 0) {
        const uint2 ua = *reinterpret_cast<const uint2*>(scA + blk0);
        const uint2 ub = *reinterpret_cast<const uint2*>(scA + 8 * nb + blk0);
        const float2 a01 = __half22float2(*reinterpret_cast<const __half2*>(&ua.x));
        const float2 a23 = __half22float2(*reinterpret_cast<const __half2*>(&ua.y));
        const float2 b01 = __half22float2(*reinterpret_cast<const __half2*>(&ub.x));
        const float2 b23 = __half22float2(*reinterpret_cast<const __half2*>(&ub.y));
        dA[0] = a01.x; dA[1] = a01.y; dA[2] = a23.x; dA[3] = a23.y;
        dB[0] = b01.x; dB[1] = b01.y; dB[2] = b23.x; dB[3] = b23.y;
    } else {
#pragma unroll
        for (int i = 0; i < GV_BPW; ++i) {
            dA[i] = __half2float(__ushort_as_half(scA[blk0 + i]));
            dB[i] = __half2float(__ushort_as_half(scA[8 * nb + blk0 + i]));
        }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const float4 c = *reinterpret_cast<const float4*>(cr + 4 * j * nbp + blk0);
        const float cv[GV_BPW] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int i = 0; i < GV_BPW; ++i) {
            if (FULL || i < nv) {
                totA[j] = fmaf(dA[i], (acc[i][j][0] + acc[i][j][1]) - cv[i], totA[j]);
                totB[j] = fmaf(dB[i], (acc[i][j][2] + acc[i][j][3]) - cv[i], totB[j]);
            }
        }
    }
}

}  // namespace

// Registers: two CTAs per SM (18 warps spread over four 16K-register
// sub-partitions) fit only at <= 96 registers a thread.  Four tokens in a
// k-split launch (64 KB of x, one CTA per SM) take 112 and two n8 tiles 128
// (with 128 KB of x).
__host__ __device__ constexpr int gv_maxnreg(int MT, int mode) {
    return gv_tiles(MT) == 2 ? 128 : (mode == GV_KSPLIT && MT == 4 ? 112 : 96);
}
template <int MT, int MODE, int NJ>
__global__ void __maxnreg__(gv_maxnreg(MT, MODE))
    tq2_gemv_kernel(const __grid_constant__ GemvTab<NJ> tab, int units, int stages, int sslots) {
    constexpr int UR = gv_unit_rows(MODE);
    constexpr int NT = gv_tiles(MT);
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ GvJobS sj[NJ];
    const GvLayout L = gv_layout(tab.K, MT, MODE, stages, sslots);
    const int njobs = tab.njobs;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + GV_MAX_STAGES;
    uint64_t* sfull = empty + GV_MAX_STAGES;
    uint64_t* sempty = sfull + GV_MAX_SSLOTS;
    float* red = reinterpret_cast<float*>(smem + L.off_red);       // [2][GV_CONS][16][MT] (k-split)
    float* corr = reinterpret_cast<float*>(smem + L.off_corr);     // [MT][nbp]
    uint8_t* scb = smem + L.off_sc;                                // [sslots] x ([UR][nb] f16)
    uint2* xs = reinterpret_cast<uint2*>(smem + L.off_xs);         // [nb][4][2MT][4][2]
    // [stages][8 warps][16 rows][128 B], 1 KB aligned for the 128-byte swizzle
    uint8_t* ring = smem + L.off_ring + ((1024u - ((smem_u32(smem) + L.off_ring) & 1023u)) & 1023u);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = L.nb, nch = L.nch, K = tab.K, Mr = tab.M;
    const int nbp = (nb + 3) & ~3;
    const int u_begin = (int)(((int64_t)blockIdx.x * units) / gridDim.x);
    const int u_end = (int)(((int64_t)(blockIdx.x + 1) * units) / gridDim.x);

    if ((int)threadIdx.x < njobs) {
        const GemvJob& J = tab.job[threadIdx.x];
        sj[threadIdx.x] = GvJobS{J.scales, J.x, J.out, J.N, J.unit0};
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], GV_CONS);
        }
        for (int s = 0; s < sslots; ++s) {
            mbar_init(&sfull[s], 1);
            mbar_init(&sempty[s], GV_CONS);
        }
        fence_mbar_init();
    }
    __syncthreads();
    // Dependents may launch now: they take SM room only where this grid
    // leaves some, and their producers stream while this grid computes.
    pdl_launch_dependents();

    // unit -> (job, first row); a CTA's units are consecutive, so the job
    // index only moves forward
    auto locate = [&](int u, int& job, int& n0) {
        while (job + 1 < njobs && u >= sj[job + 1].unit0) ++job;
        n0 = (u - sj[job].unit0) * UR;
    };

    if (warp == GV_CONS) {
        // ------------------------------------------------ producer warp ----
        if (lane != 0) return;
        int it = 0, job = 0, s = 0, slot = 0;
        uint32_t ph = 0, sph = 0;                // phase parity of the current ring / slot round
        bool ok = true;
        for (int u = u_begin, ui = 0; u < u_end && ok; ++u, ++ui) {
            int n0;
            locate(u, job, n0);
            const GvJobS& J = sj[job];
            const int rows = min(UR, J.N - n0);
            if (ui >= sslots) ok = mbar_wait(&sempty[slot], sph ^ 1u);
            if (!ok) break;
            // rounded up to 16 bytes: the scale plane carries 16 bytes of padding
            const uint32_t sbytes = ((uint32_t)rows * nb * 2 + 15u) & ~15u;
            mbar_arrive_expect_tx(&sfull[slot], sbytes);
            bulk_load(scb + slot * L.sc_bytes, J.scales + (int64_t)n0 * nb, sbytes, &sfull[slot]);
            if (++slot == sslots) { slot = 0; sph ^= 1u; }
            // row-split consumers take the pieces partial-major (c = j, j + 8,
            // ... for j = 0..7); k-split consumers in order
            for (int i = 0, c = 0, j = 0; i < nch; ++i, ++it) {
                if (it >= stages) ok = mbar_wait(&empty[s], ph ^ 1u);
                if (!ok) break;
                mbar_arrive_expect_tx(&full[s], (uint32_t)GV_STAGE);
                tma_load_3d(ring + s * GV_STAGE, &tab.job[job].map, &full[s], 0, n0,
                            MODE == GV_ROWS ? c : c * GV_CONS);
                if (++s == stages) { s = 0; ph ^= 1u; }
                if (MODE == GV_ROWS) {
                    c += GV_CONS;
                    if (c >= nch) c = ++j;
                } else {
                    ++c;
                }
            }
        }
        return;
    }

    // ---------------------------------------------------- consumer warps ----
    const int g = lane >> 2, t = lane & 3;
    const int tm = t < MT ? t : MT - 1;          // token of this lane's D columns 2t, 2t+1 in tile 0 (if t < MT)
    const float* cr = corr + tm * nbp;
    // staging role of this lane: block (lane / 8) of the pass, word pair t, half y
    const int st_q = lane >> 3, st_t = (lane >> 1) & 3, st_y = lane & 1;
    // x blocks this warp converts: k-split -- the ones it uses,
    // c * 32 + 4 * warp + i, listed c-major; row-split -- warp, warp + 8, ...
    int nbw = 0;
    if (MODE == GV_KSPLIT) {
#pragma unroll
        for (int i = 0; i < GV_BPW; ++i) {
            const int r = nb - GV_BPW * warp - i;
            nbw += r > 0 ? (r + GV_BPW * GV_CONS - 1) / (GV_BPW * GV_CONS) : 0;
        }
    } else {
        nbw = nb > warp ? (nb - warp + GV_CONS - 1) / GV_CONS : 0;
    }
    auto consumers_sync = [] { asm volatile("bar.sync 1, %0;" ::"n"(GV_CONS * 32) : "memory"); };

    // this lane's x fragments (uint4 units); lanes g >= 2MT alias column g % 2MT
    const int xstep = 4 * (2 * MT) * 4, sstep = (2 * MT) * 4;
    const uint4* xl = reinterpret_cast<const uint4*>(xs) + (g % (2 * MT)) * 4 + t;
    const uint32_t z = (uint32_t)(K >> 30);      // 0 (K < 2^30), opaque to the compiler
    const GvShift sh{16u | z, (1u << 26) | z, 0x00300030u | z, 0x00C000C0u | z, 0x03000300u | z};
    // A fragments of a word whose 16 codes are all 1 (weight 0), k16 steps 0..3
    uint32_t ones[4][4];
    {
        uint32_t w1[3];
        gv_word(0x55555555u | z, sh, w1);
        gv_afrag<0>(w1, w1, ones[0], sh);
        gv_afrag<1>(w1, w1, ones[1], sh);
        gv_afrag<2>(w1, w1, ones[2], sh);
        gv_afrag<3>(w1, w1, ones[3], sh);
    }

    pdl_wait();
    const float* staged = nullptr;
    auto stage_x = [&](const float* x) {
        if (MODE == GV_ROWS && staged) consumers_sync();     // everyone is done with the old x
        for (int p = 0; p < (nbw + 3) / 4; ++p) {
            const int li = 4 * p + st_q;                      // index in this warp's block list
            const bool live = li < nbw;                       // uniform within each 8-lane group
            const int blk = MODE == GV_KSPLIT ? (li / GV_BPW) * (GV_BPW * GV_CONS) + GV_BPW * warp + li % GV_BPW
                                              : warp + GV_CONS * li;
            const int k0 = (live ? blk : 0) * 128 + 32 * st_t + 16 * st_y;
            // tokens in batches of SB: all of a batch's loads are issued
            // before any is converted, so a batch costs one L2 round trip
            constexpr int SB = MT == 8 && MODE == GV_KSPLIT ? 4 : (MT >= 2 && gv_maxnreg(MT, MODE) > 96 ? 2 : 1);
#pragma unroll
            for (int m0 = 0; m0 < MT; m0 += SB) {
                float4 q[SB][4];
#pragma unroll
                for (int mb = 0; mb < SB; ++mb) {
                    const int m = m0 + mb;
                    const float4* src = reinterpret_cast<const float4*>(x + (int64_t)m * K + k0);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        q[mb][v] = live && m < Mr ? __ldg(src + v) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                if (live) {
#pragma unroll
                    for (int mb = 0; mb < SB; ++mb) {
                        const int m = m0 + mb;
                        const float e[16] = {q[mb][0].x, q[mb][0].y, q[mb][0].z, q[mb][0].w,
                                             q[mb][1].x, q[mb][1].y, q[mb][1].z, q[mb][1].w,
                                             q[mb][2].x, q[mb][2].y, q[mb][2].z, q[mb][2].w,
                                             q[mb][3].x, q[mb][3].y, q[mb][3].z, q[mb][3].w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {           // k16 step 4y + j: pairs 2j, 2j+1
                            uint32_t h01, l01, h23, l23;
                            split2(e[2 * j], e[2 * j + 8], h01, l01);
                            split2(e[2 * j + 1], e[2 * j + 9], h23, l23);
                            // step 4y + j -> pair 2y + j/2, half j % 2
                            uint2* d = xs + (((blk * 4 + 2 * st_y + (j >> 1)) * (2 * MT) + 2 * m) * 4 + st_t) * 2 + (j & 1);
                            d[0] = make_uint2(h01, h23);          // column 2m: hi
                            d[8] = make_uint2(l01, l23);          // column 2m+1: lo
                        }
                    }
                }
            }
        }
        if (MODE == GV_ROWS) consumers_sync();                // every block converted
        else __syncwarp();
        // Corrections sum_k (m_q+1) x_k per block and token: the MMA chain of
        // gv_piece (same steps, same order, accumulator from zero) on a row of
        // all code-1 weights, so that d * (acc - correction) is exactly 0 for
        // such a block.  Each warp takes the blocks it staged, CI chains at a
        // time, interleaved (fewer where registers are scarce).
        constexpr int CI = MT >= 2 && gv_maxnreg(MT, MODE) <= 96 ? (MODE == GV_KSPLIT ? 1 : 2) : 4;
        for (int l0 = 0; l0 < nbw; l0 += CI) {
            int blk[CI];
            float acc[CI][NT][4];
#pragma unroll
            for (int i = 0; i < CI; ++i) {
                const int li = min(l0 + i, nbw - 1);              // past the end: repeat the last block
                blk[i] = MODE == GV_KSPLIT ? (li / GV_BPW) * (GV_BPW * GV_CONS) + GV_BPW * warp + li % GV_BPW
                                           : warp + GV_CONS * li;
#pragma unroll
                for (int j = 0; j < NT; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.f;
            }
#pragma unroll
            for (int p = 0; p < 4; ++p) {
#pragma unroll
                for (int i = 0; i < CI; ++i) {
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const uint4 b = xl[blk[i] * xstep + p * sstep + 32 * j];
                        mma_16816_pure(acc[i][j], ones[(2 * p) & 3], b.x, b.y);
                        mma_16816_pure(acc[i][j], ones[(2 * p + 1) & 3], b.z, b.w);
                    }
                }
            }
            if (g == 0 && t < MT) {
#pragma unroll
                for (int i = 0; i < CI; ++i)
#pragma unroll
                    for (int j = 0; j < NT; ++j) corr[(t + 4 * j) * nbp + blk[i]] = acc[i][j][0] + acc[i][j][1];
            }
        }
        if (MODE == GV_ROWS) consumers_sync();                // every correction written
        else __syncwarp();
        staged = x;
    };

    int s = 0, slot = 0, job = 0;
    uint32_t ph = 0, sph = 0;
    bool dead = false;                            // a bounded wait ran out: skip the rest
    const int rbase = MODE == GV_ROWS ? 16 * warp : 0;
    for (int u = u_begin; u < u_end; ++u) {
        int n0;
        locate(u, job, n0);
        const GvJobS& J = sj[job];
        if (J.x != staged) stage_x(J.x);
        if (!dead && !mbar_wait(&sfull[slot], sph)) dead = true;
        const uint16_t* scA = reinterpret_cast<const uint16_t*>(scb + slot * L.sc_bytes) + (rbase + g) * nb;
        auto do_stage = [&](int c, float (&ta)[NT], float (&tb)[NT]) {
            if (!dead && !mbar_wait(&full[s], ph)) dead = true;   // after a timeout: no more waits
            const uint8_t* pc = ring + s * GV_STAGE + warp * GV_WARP_BYTES + g * GV_PIECE + 8 * (t & 1);
            const int blk0 = MODE == GV_ROWS ? GV_BPW * c : c * (GV_BPW * GV_CONS) + GV_BPW * warp;
            const int nv = min(GV_BPW, nb - blk0);              // valid blocks (warp-uniform)
            if (nv == GV_BPW) gv_piece<MT, true>(pc, g, t, xl, xstep, sstep, cr, nbp, blk0, nv, nb, scA, sh, ta, tb);
            else if (nv > 0) gv_piece<MT, false>(pc, g, t, xl, xstep, sstep, cr, nbp, blk0, nv, nb, scA, sh, ta, tb);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            if (++s == stages) { s = 0; ph ^= 1u; }
        };
        float totA[NT], totB[NT];                // rows rbase+g and rbase+g+8; tokens tm, tm + 4
#pragma unroll
        for (int j = 0; j < NT; ++j) totA[j] = totB[j] = 0.f;
        if (MODE == GV_KSPLIT) {
            for (int c = 0; c < nch; ++c) do_stage(c, totA, totB);
        } else {
            // Eight partial sums, one per piece index mod 8, taken one after
            // the other (the producer loads the pieces in this order): the
            // blocks of partial j are exactly those warp j owns in a k-split
            // launch, in the same order, and the partials are added in the
            // same order as the k-split reduction.  One partial pair is live
            // at a time instead of eight.
            for (int j = 0; j < GV_CONS; ++j) {
                float pa[NT], pb[NT];
#pragma unroll
                for (int q = 0; q < NT; ++q) pa[q] = pb[q] = 0.f;
                for (int c = j; c < nch; c += GV_CONS) do_stage(c, pa, pb);
#pragma unroll
                for (int q = 0; q < NT; ++q) {
                    totA[q] += pa[q];
                    totB[q] += pb[q];
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sempty[slot]);
        const int ui = u - u_begin;
        if (++slot == sslots) { slot = 0; sph ^= 1u; }

        if (MODE == GV_ROWS) {
            if (t < MT) {
                const int ra = n0 + rbase + g;
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const int m = t + 4 * j;
                    if (m < Mr) {
                        if (ra < J.N) J.out[(int64_t)m * J.N + ra] = totA[j];
                        if (ra + 8 < J.N) J.out[(int64_t)m * J.N + ra + 8] = totB[j];
                    }
                }
            }
        } else {
            float* rd = red + (ui & 1) * (GV_CONS * 16 * MT);
            if (t < MT) {
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    rd[(warp * 16 + g) * MT + t + 4 * j] = totA[j];
                    rd[(warp * 16 + g + 8) * MT + t + 4 * j] = totB[j];
                }
            }
            consumers_sync();
            if ((int)threadIdx.x < 16 * MT) {
                const int m = threadIdx.x >> 4, r = threadIdx.x & 15;
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < GV_CONS; ++w) sum += rd[(w * 16 + r) * MT + m];
                if (m < Mr && n0 + r < J.N) J.out[(int64_t)m * J.N + n0 + r] = sum;
            }
        }
    }
}

namespace {

// Ring depth and scale slots: with `pair`, as many stages as fit beside a
// second CTA (false below four), else all of an SM's shared memory.
// Row-split grids put two of their own CTAs on an SM; k-split grids put one
// CTA on every SM and take the pair budget when it leaves four stages, so
// the next kernel's CTA (launched early) fits beside it on every SM and
// streams its weights meanwhile (chained 4096^2 GEMVs 4.9 -> 4.8 us; with a
// grid that left SMs idle the early CTAs doubled up there and ran slower).
// Enough scale slots that the code ring, not the scales, limits how far the
// producer runs ahead.  False if nothing fits.
bool gv_plan(int K, int MT, int mode, bool pair, int& stages, int& sslots) {
    sslots = 2;
    for (int pass = 0; pass < 2; ++pass) {
        const int fixed = (int)gv_layout(K, MT, mode, 0, sslots).total;
        stages = ((pair ? GV_SMEM_PAIR : GV_SMEM_MAX) - fixed) / GV_STAGE;
        if (stages > GV_MAX_STAGES) stages = GV_MAX_STAGES;
        if (stages < (pair ? 4 : 2)) return false;
        if (pass == 0) {
            const int nch = (K / 128 + gv_stage_blocks(mode) - 1) / gv_stage_blocks(mode);
            sslots = (stages + nch - 1) / nch + 1;
            if (sslots > GV_MAX_SSLOTS) sslots = GV_MAX_SSLOTS;
        }
    }
    return true;
}

template <int MT, int MODE, int NJ>
cudaError_t gv_launch(const GemvTab<NJ>& tab, int units, int stages, int sslots, int sms, int dev,
                      cudaStream_t st) {
    static bool configured[64] = {false};
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(tq2_gemv_kernel<MT, MODE, NJ>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, GV_SMEM_MAX);
        // row-split: ask for the largest shared-memory carveout so that two
        // CTAs fit on an SM (the default picks one just large enough for one)
        if (e == cudaSuccess && MODE == GV_ROWS)
            e = cudaFuncSetAttribute(tq2_gemv_kernel<MT, MODE, NJ>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    // two CTAs per SM where the plan leaves room (eight consumer warps alone
    // do not hide the MMA and load latency), else one; every slot gets work
    // (units split as evenly as the count allows), so no SM is left for the
    // next kernel's early CTAs to double up on
    const GvLayout L = gv_layout(tab.K, MT, MODE, stages, sslots);
    const bool pair = L.total + 2048u <= (uint32_t)GV_SMEM_PAIR && gv_maxnreg(MT, MODE) <= 96;   // two CTAs fit
    const int slots = pair ? 2 * sms : sms;
    const int grid = units < slots ? units : slots;
    return launch_pdl(tq2_gemv_kernel<MT, MODE, NJ>, dim3((unsigned)grid), dim3(GV_THREADS), (size_t)L.total, st,
                      tab, units, stages, sslots);
}

template <int NJ>
cudaError_t gv_dispatch(const tq2_weight* const* ws, const float* const* xs, float* const* outs, int G, int M,
                        cudaStream_t st) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int K = (int)ws[0]->K;
    int64_t units_r = 0;
    for (int g = 0; g < G; ++g) units_r += (ws[g]->N + gv_unit_rows(GV_ROWS) - 1) / gv_unit_rows(GV_ROWS);
    const int MT = gv_mt(M);
    int stages = 0, sslots = 0;
    int mode = GV_KSPLIT;
    // row-split (two CTAs per SM where they fit) when its units fill the
    // GPU; else k-split, one CTA per SM (two per SM measured no faster for
    // single calls), within the pair budget when four stages fit there
    if (units_r >= sms && (gv_plan(K, MT, GV_ROWS, true, stages, sslots) ||
                           gv_plan(K, MT, GV_ROWS, false, stages, sslots)))
        mode = GV_ROWS;
    else if (!gv_plan(K, MT, GV_KSPLIT, true, stages, sslots) && !gv_plan(K, MT, GV_KSPLIT, false, stages, sslots))
        return cudaErrorInvalidValue;

    GemvTab<NJ> tab;
    tab.njobs = G;
    tab.K = K;
    tab.M = M;
    int64_t units = 0;
    for (int g = 0; g < G; ++g) {
        const tq2_weight* w = ws[g];
        tab.job[g].map = mode == GV_ROWS ? w->gemv_map_r : w->gemv_map_k;
        tab.job[g].scales = w->scales;
        tab.job[g].x = xs[g];
        tab.job[g].out = outs[g];
        tab.job[g].N = (int)w->N;
        tab.job[g].unit0 = (int)units;
        units += (w->N + gv_unit_rows(mode) - 1) / gv_unit_rows(mode);
    }
#define GV_LAUNCH(T)                                                                     \
    return mode == GV_ROWS ? gv_launch<T, GV_ROWS>(tab, (int)units, stages, sslots, sms, dev, st) \
                           : gv_launch<T, GV_KSPLIT>(tab, (int)units, stages, sslots, sms, dev, st)
    switch (MT) {
        case 1: GV_LAUNCH(1);
        case 2: GV_LAUNCH(2);
        case 4: GV_LAUNCH(4);
        default: GV_LAUNCH(8);
    }
#undef GV_LAUNCH
}

bool make_map(tq2_weight* w, CUtensorMap* map, uint32_t rows, uint32_t pieces) {
    const uint64_t npieces = (uint64_t)(w->K / 4 + GV_PIECE - 1) / GV_PIECE;
    const uint64_t dims[3] = {(uint64_t)GV_PIECE, (uint64_t)w->N, npieces};
    const uint64_t strides[2] = {(uint64_t)(w->K / 4), (uint64_t)GV_PIECE};
    const uint32_t box[3] = {(uint32_t)GV_PIECE, rows, pieces};
    return make_tensor_map_3d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, w->codes, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

bool gemv_supports(int M, int64_t K) {
    return M >= 1 && M <= GEMV_MAX_M && K >= 128 && (int64_t)gv_mt(M) * K <= GEMV_MAX_MK;
}

bool make_gemv_maps(tq2_weight* w) {
    return make_map(w, &w->gemv_map_k, 16u, (uint32_t)GV_CONS) &&
           make_map(w, &w->gemv_map_r, (uint32_t)gv_unit_rows(GV_ROWS), 1u);
}

cudaError_t launch_gemv(const tq2_weight* const* ws, const float* const* xs, float* const* outs, int G, int M,
                        cudaStream_t st) {
    if (G < 1 || G > GEMV_MAX_JOBS || !gemv_supports(M, ws[0]->K)) return cudaErrorInvalidValue;
    if (G == 1) return gv_dispatch<1>(ws, xs, outs, G, M, st);
    return gv_dispatch<GEMV_MAX_JOBS>(ws, xs, outs, G, M, st);
}

unsigned int read_clear_dev_error_gemv(cudaStream_t st) {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_dev_error, sizeof(v), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return 0;
    cudaMemcpyToSymbolAsync(g_dev_error, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
    cudaStreamSynchronize(st);
    return v;
}

}  // namespace tq2
