// blr_rank.cu -- the rank-space products of the binary low-rank layer
// ("cortiq-engine 0.8.43, src/gpu_wgpu/train_mm.rs", blr_forward and
// blr_backward):
//
//   forward   a[t,k] = sum_j (x[t,j] g[j]) S_V[j,k]               (K = d_in)
//   backward  b[t,k] = sum_i (dy[t,i] h[i] gs) S_U[i,k] / gs       (K = d_out)
//
// as one pass over the f32 activations: the activation is read once from
// HBM, scaled and rounded to f16 on chip, and multiplied by the sign plane on
// the tensor cores; nothing but the [T][r] results goes back to memory.
//
// One CTA computes a 128-token x RB-rank tile (RB = 256, or 128 when r is
// not a multiple of 256) over a slice of K; the CL CTAs of a cluster take
// the CL slices of the same tile and add their partial sums through
// distributed shared memory in a fixed order (deterministic).  Roles:
//   * one thread streams each stage's operands into shared memory: the f32
//     activation tile (128 tokens x 64, two 32-column TMA boxes, 128-byte
//     swizzle), the stage's 64 rows of sign words for the CTA's ranks (TMA)
//     and the stage's 64 column factors (bulk copy);
//   * eight converter warps (two per 32-token lane quarter, one per 32-column
//     half of a stage) read their token's activations of every stage from
//     there, multiply by the column vector and the scale, round to f16 and
//     store them into a ring in tensor memory: the MMA's A operand (tokens =
//     M = 128 lanes);
//   * four decoder warps expand the stage's 64 sign rows (the plane's row
//     index is the GEMM's K) into the MMA's B operand in shared memory,
//     MN-major (ranks contiguous) with 128-byte swizzling, so the bitmap is
//     read in its own row order and never transposed; set bit -> +1.0,
//     clear -> -1.0;
//   * one warp issues tcgen05.mma (kind::f16, A from tensor memory, B from
//     shared memory, f32 accumulation in tensor memory, N = RB);
//   * after a cluster barrier (every CTA's main loop is done, so every ring
//     may be overwritten) the decoder warps drain the accumulator and store
//     each row straight into the shared memory of the CTA that owns it (CTA z
//     owns rows [z*128/CL, (z+1)*128/CL) of the tile), into a slot of its
//     inbox per source CTA; after a second cluster barrier each CTA sums its
//     inbox over the CL sources in a fixed order and writes the result, its
//     f16 staging for the next GEMM, and (backward) the per-32-token partial
//     column sums of result * other.
// Within each 64-rank group the B operand holds ranks in the order the bits
// fall out of a word: MN element 2p + h of the group is rank
// (p < 16 ? 0 : 32) + p % 16 + 16 h.  That is also the order in which the
// next GEMM (the core's DecSign decoder) expects its f16 operand inside every
// 32-rank group, so the staged f16 row is the accumulator row as it stands.
#include "tq2_internal.h"
#include "umma_core.cuh"

namespace tq2 {

namespace {

constexpr int BR_THREADS = 512;
constexpr int BR_BK = 64;              // K per stage
constexpr int BR_MAX_STAGES = 8;

struct BrBars {
    uint64_t xfull[BR_MAX_STAGES];   // a stage's activations, sign words and column factors landed
    uint64_t xempty[BR_MAX_STAGES];  // ... and have been read (8 converter + 4 decoder warps)
    uint64_t full[BR_MAX_STAGES];    // a stage's A (8 converter warps) and B (4 decoder warps) are written
    uint64_t empty[BR_MAX_STAGES];
    uint64_t acc_full;
    uint32_t tmem_base;
    int abort;
};

struct BrArgs {
    const float* act;          // [T][K] f32
    const float* vec;          // [K] column factors of the activation
    float scale;               // power of two multiplying the staged activation
    const uint32_t* bits;      // [K][r/32], row j = plane row j (the GEMM's K index)
    int T, K, r;
    float oscale;              // result = accumulator * oscale
    float* res;                // [T][r] f32 result, or null
    const float* col;          // [r] factor of the f16 staging
    float scale2;              // power of two of the f16 staging
    uint16_t* st16;            // [T][r] f16 of result * col * scale2, 32-group pair order
    const float* other;        // [T][r] or null: column sums of result * other
    float* colpart;            // [T/32 chunks][r] partial column sums (rows of 32 tokens)
};

// rank offset inside a 64-rank group of MN element n (0..63)
__device__ __forceinline__ int br_rank_of(int n) {
    const int p = n >> 1, h = n & 1;
    return (p < 16 ? 0 : 32) + (p & 15) + 16 * h;
}

}  // namespace

template <int RB>
__global__ void __launch_bounds__(BR_THREADS, 1) blr_rank_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                 const __grid_constant__ CUtensorMap bmap,
                                                                 const BrArgs A, int S, int CL) {
    constexpr int STAGE_B = BR_BK * RB * 2;                 // B stage bytes (64 K rows x RB ranks f16)
    constexpr int STAGE_X = BR_BK * 128 * 4;                // activation stage bytes (128 tokens x 64 f32)
    constexpr int STAGE_W = BR_BK * (RB / 32) * 4;          // sign words of a stage (64 rows x RB/32 words)
    constexpr int STAGE_G = BR_BK * 4;                      // column factors of a stage
    constexpr int NA = RB / 64;                             // MN atoms a stage
    constexpr int RED_LD = RB + 4;                          // padded row of the drained partial (floats)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* bring = smem;                                  // [S][STAGE_B] sign-plane operand
    uint8_t* xring = smem + S * STAGE_B;                    // [S][STAGE_X] activation tiles
    uint8_t* wring = xring + S * STAGE_X;                   // [S][STAGE_W] sign words
    float* gring = reinterpret_cast<float*>(wring + S * STAGE_W);   // [S][64] column factors
    const int used = S * (STAGE_B + STAGE_X + STAGE_W + STAGE_G);
    const int ring_bytes = used > 128 * RED_LD * 4 ? used : 128 * RED_LD * 4;
    BrBars* bars = reinterpret_cast<BrBars*>(smem + ring_bytes + 16384);   // 16 KB guard after the rings
    float* red = reinterpret_cast<float*>(smem);            // inbox [CL][128/CL][RED_LD], after the main loops

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int z = (int)cluster_ctarank();                   // K slice = rank in the cluster
    const int rb = blockIdx.y, tile = blockIdx.z;
    const int nk = A.K / BR_BK;
    const int k0 = (int)(((int64_t)nk * z) / CL), k1 = (int)(((int64_t)nk * (z + 1)) / CL);
    const int nst = k1 - k0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&bars->xfull[s], 1);
            mbar_init(&bars->xempty[s], 12);
            mbar_init(&bars->full[s], 12);
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->acc_full, 1);
        bars->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&xmap);
        tma_prefetch_desc(&bmap);
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, 512u);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t a_col0 = (uint32_t)RB;                   // A ring after the accumulator
    volatile int* abort_flag = &bars->abort;
    pdl_launch_dependents();

    if (warp == 0) {
        // ---- MMA issuer: the whole warp waits (one barrier a stage), the next
        // stage's barrier is tested without blocking before this stage's MMAs,
        // and an elected lane issues; the tensor pipe idles whenever this warp
        // spends time between stages.
        const uint32_t idesc = idesc_f16_f32_bmn(128, (uint32_t)RB);
        int s = 0;
        uint32_t ph = 0;
        bool ok = true, ready = false;
        for (int i = 0; i < nst; ++i) {
            if (!ready && !__all_sync(0xffffffffu, mbar_wait_or_abort(&bars->full[s], ph, abort_flag, true))) {
                *abort_flag = 1;
                ok = false;
                break;
            }
            const int s1 = s + 1 == S ? 0 : s + 1;
            const uint32_t ph1 = s + 1 == S ? ph ^ 1u : ph;
            ready = i + 1 < nst && mbar_test_wait(&bars->full[s1], ph1);
            tc_fence_after();
            const uint32_t bbase = smem_u32(bring + s * STAGE_B);
            const uint32_t acol = tmem + a_col0 + (uint32_t)(s * (BR_BK / 2));
#pragma unroll
            for (int j = 0; j < BR_BK / 16; ++j) {
                // k16 step j = K atoms 2j, 2j+1 (each NA * 1024 bytes)
                const uint64_t bdesc = sdesc_mnmajor_sw128(bbase + (uint32_t)(j * 2 * NA * 1024), 1024u,
                                                           (uint32_t)(NA * 1024));
                umma_f16_ts_elect(tmem, acol + (uint32_t)(j * 8), bdesc, idesc, (i > 0 || j > 0) ? 1u : 0u);
            }
            umma_commit_elect(&bars->empty[s]);
            s = s1;
            ph = ph1;
            ready = __all_sync(0xffffffffu, ready);
        }
        if (ok && nst > 0) {
            umma_commit_elect(&bars->acc_full);
            // every MMA must have finished reading this CTA's rings before the
            // cluster barrier lets peers store into them
            mbar_wait_or_abort(&bars->acc_full, 0u, abort_flag, true);
        }
    } else if (warp == 2) {
        // ---- TMA producer of the activation tiles
        if (lane == 0) {
            pdl_wait();
            for (int i = 0; i < nst; ++i) {
                const int s = i % S;
                const uint32_t ph = (uint32_t)(i / S) & 1u;
                if (i >= S && !mbar_wait_or_abort(&bars->xempty[s], ph ^ 1u, abort_flag)) {
                    *abort_flag = 1;
                    break;
                }
                mbar_arrive_expect_tx(&bars->xfull[s], (uint32_t)(STAGE_X + STAGE_W + STAGE_G));
                const int kx = (k0 + i) * BR_BK;
                tma_load_2d(xring + s * STAGE_X, &xmap, &bars->xfull[s], kx, tile * 128);
                tma_load_2d(xring + s * STAGE_X + STAGE_X / 2, &xmap, &bars->xfull[s], kx + 32, tile * 128);
                tma_load_2d(wring + s * STAGE_W, &bmap, &bars->xfull[s], rb * (RB / 32), kx);
                bulk_load(gring + s * BR_BK, A.vec + kx, (uint32_t)STAGE_G, &bars->xfull[s]);
            }
        }
    } else if (warp >= 4 && warp < 12) {
        // ---- converters: token row 32q + lane of the tile, columns 32h..32h+31
        // of every stage (box h of the stage's activation tile).  Every
        // converter warp takes every stage, so no warp can run a ring round
        // ahead of another: a wait on a phase parity is never ambiguous.
        const int q = warp & 3, h = (warp - 4) >> 2;
        const int i_row = q * 32 + lane;
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + a_col0 + (uint32_t)(16 * h);
        for (int i = 0; i < nst; ++i) {
            const int s = i % S;
            const uint32_t ph = (uint32_t)(i / S) & 1u;
            if (!mbar_wait_or_abort(&bars->xfull[s], ph, abort_flag)) {
                *abort_flag = 1;
                break;
            }
            // row i_row of box h: 16-byte chunk c (columns 32h + 4c..) at chunk c ^ (i_row & 7)
            // The slot goes back to the TMA producer only after the values read
            // from it have been used, and after a proxy fence: the next write
            // into it comes through the async proxy.
            uint32_t w[16];
            const uint8_t* xr = xring + s * STAGE_X + h * (STAGE_X / 2) + i_row * 128;
            const float4* vv = reinterpret_cast<const float4*>(gring + s * BR_BK + 32 * h);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 v = *reinterpret_cast<const float4*>(xr + ((c ^ (i_row & 7)) << 4));
                const float4 g = vv[c];
                const __half2 lo = __floats2half2_rn(v.x * g.x * A.scale, v.y * g.y * A.scale);
                const __half2 hi = __floats2half2_rn(v.z * g.z * A.scale, v.w * g.w * A.scale);
                w[2 * c] = *reinterpret_cast<const uint32_t*>(&lo);
                w[2 * c + 1] = *reinterpret_cast<const uint32_t*>(&hi);
            }
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->xempty[s]);
            if (i >= S && !mbar_wait_or_abort(&bars->empty[s], ph ^ 1u, abort_flag)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            tmem_st_32x32b_x16(taddr + (uint32_t)(s * (BR_BK / 2)), w);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->full[s]);
        }
    } else if (warp >= 12) {
        // ---- decoders of the sign plane, then the accumulator drain
        const int q = warp & 3, tid = q * 32 + lane;      // 0..127
        constexpr int ITEMS = BR_BK * NA;                   // (row, 64-rank group) items a stage
        for (int i = 0; i < nst; ++i) {
            const int s = i % S;
            const uint32_t ph = (uint32_t)(i / S) & 1u;
            if (!mbar_wait_or_abort(&bars->xfull[s], ph, abort_flag)) {
                *abort_flag = 1;
                break;
            }
            // item it = row j (fastest, so the 8 lanes of a 16-byte store phase
            // write 8 different rows: 8 bank groups) x 64-rank group na
            uint2 wv[ITEMS / 128];
            const uint32_t* wst = reinterpret_cast<const uint32_t*>(wring + s * STAGE_W);
#pragma unroll
            for (int u = 0; u < ITEMS / 128; ++u) {
                const int it = tid + 128 * u, j = it % BR_BK, na = it / BR_BK;
                wv[u] = *reinterpret_cast<const uint2*>(wst + j * (RB / 32) + 2 * na);
            }
            fence_proxy_async_shared();                     // the slot is refilled through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->xempty[s]);
            if (i >= S && !mbar_wait_or_abort(&bars->empty[s], ph ^ 1u, abort_flag)) {
                *abort_flag = 1;
                break;
            }
            uint8_t* stage = bring + s * STAGE_B;
#pragma unroll
            for (int u = 0; u < ITEMS / 128; ++u) {
                const int it = tid + 128 * u, j = it % BR_BK, na = it / BR_BK;
                uint32_t c[32];
                DecSign::word(wv[u].x, c);
                DecSign::word(wv[u].y, c + 16);
                // atom (K atom j/8, MN atom na), row j%8; chunk cc at cc ^ (j%8)
                uint8_t* row = stage + (j >> 3) * (NA * 1024) + na * 1024 + (j & 7) * 128;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)
                    *reinterpret_cast<uint4*>(row + ((cc ^ (j & 7)) << 4)) =
                        make_uint4(c[4 * cc], c[4 * cc + 1], c[4 * cc + 2], c[4 * cc + 3]);
            }
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->full[s]);
        }
    }

    // every CTA of the cluster is past its main loop: the rings may be reused
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    const int RPC = 128 / CL;                               // CL in {1, 2, 4}: a multiple of 32
    if (warp >= 12) {
        // drain: TMEM lane 32q + lane = token row of the tile, pushed to the
        // owner CTA's inbox slot of this CTA (local when this CTA owns it)
        const int q = warp & 3, row = q * 32 + lane;
        const int owner = row / RPC, lr = row % RPC;
        const uint32_t dst = mapa_shared(smem_u32(red + (z * RPC + lr) * RED_LD), (uint32_t)owner);
        const bool have = nst > 0 && mbar_wait_or_abort(&bars->acc_full, 0u, abort_flag);
        if (have) tc_fence_after();
        const uint32_t laddr = tmem + ((uint32_t)(q * 32) << 16);
        for (int cc = 0; cc < RB; cc += 32) {
            uint32_t v[32];
            if (have) {
                tmem_ld_32x32b_x32(laddr + (uint32_t)cc, v);
                tmem_wait_ld();
            } else {                                        // no stage in this slice (or a wait gave up)
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0u;
            }
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4)
                st_dsmem_f4(dst + (uint32_t)((cc + 4 * i4) * 4),
                            make_float4(__uint_as_float(v[4 * i4]), __uint_as_float(v[4 * i4 + 1]),
                                        __uint_as_float(v[4 * i4 + 2]), __uint_as_float(v[4 * i4 + 3])));
        }
    }

    // every row is in its owner's inbox
    tc_fence_before();
    __syncthreads();
    cluster_sync();

    pdl_wait();                                             // col, other: earlier work on the stream
    {
        constexpr int NSEG = RB / 16;
        constexpr int NGRP = 16 / NSEG;
        const int seg = warp % NSEG, rgrp = warp / NSEG;
        const int n0 = seg * 16;                            // first accumulator column
        // the segment's 16 columns: ranks kA..kA+7 (even columns) and kA+16..kA+23 (odd)
        const int kA = rb * RB + (n0 >> 6) * 64 + br_rank_of(n0 & 63);
        // the segment's column factors (ranks kA..kA+7, kA+16..kA+23)
        float colv[16];
        {
            const float4 c0 = *reinterpret_cast<const float4*>(A.col + kA);
            const float4 c1 = *reinterpret_cast<const float4*>(A.col + kA + 4);
            const float4 c2 = *reinterpret_cast<const float4*>(A.col + kA + 16);
            const float4 c3 = *reinterpret_cast<const float4*>(A.col + kA + 20);
            const float cl[16] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w,
                                  c2.x, c2.y, c2.z, c2.w, c3.x, c3.y, c3.z, c3.w};
#pragma unroll
            for (int i = 0; i < 16; ++i) colv[i] = cl[(i >> 1) + 8 * (i & 1)];
        }
        for (int p = 0; rgrp * 32 + p * 32 * NGRP < RPC; ++p) {
            const int lr = rgrp * 32 + p * 32 * NGRP + lane;     // row of this CTA's share
            const int row = z * RPC + lr;
            const int t = tile * 128 + row;
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.f;
            for (int zz = 0; zz < CL; ++zz) {                   // sources in order
                const float4* src = reinterpret_cast<const float4*>(red + (zz * RPC + lr) * RED_LD + n0);
#pragma unroll
                for (int i4 = 0; i4 < 4; ++i4) {
                    const float4 f = src[i4];
                    v[4 * i4] += f.x; v[4 * i4 + 1] += f.y; v[4 * i4 + 2] += f.z; v[4 * i4 + 3] += f.w;
                }
            }
            const bool live = t < A.T;
            const int64_t rowoff = (int64_t)(live ? t : 0) * A.r;
            float cs[16], oth[16];
            if (A.other && live) {
                const float4 o0 = *reinterpret_cast<const float4*>(A.other + rowoff + kA);
                const float4 o1 = *reinterpret_cast<const float4*>(A.other + rowoff + kA + 4);
                const float4 o2 = *reinterpret_cast<const float4*>(A.other + rowoff + kA + 16);
                const float4 o3 = *reinterpret_cast<const float4*>(A.other + rowoff + kA + 20);
                const float ol[16] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w,
                                      o2.x, o2.y, o2.z, o2.w, o3.x, o3.y, o3.z, o3.w};
#pragma unroll
                for (int i = 0; i < 16; ++i) oth[i] = ol[(i >> 1) + 8 * (i & 1)];
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) oth[i] = 0.f;
            }
            __align__(16) uint16_t h16[16];
            __align__(16) float r0[8], r1[8];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float val = v[i] * A.oscale;
                if (i & 1) r1[i >> 1] = val; else r0[i >> 1] = val;
                h16[i] = __half_as_ushort(__float2half_rn(val * colv[i] * A.scale2));
                cs[i] = val * oth[i];
            }
            if (live) {
                if (A.res) {
                    float4* d0 = reinterpret_cast<float4*>(A.res + rowoff + kA);
                    float4* d1 = reinterpret_cast<float4*>(A.res + rowoff + kA + 16);
                    d0[0] = *reinterpret_cast<const float4*>(r0);
                    d0[1] = *reinterpret_cast<const float4*>(r0 + 4);
                    d1[0] = *reinterpret_cast<const float4*>(r1);
                    d1[1] = *reinterpret_cast<const float4*>(r1 + 4);
                }
                // staged f16: the accumulator's column order is the 32-group pair order
                uint4* dst = reinterpret_cast<uint4*>(A.st16 + rowoff + rb * RB + n0);
                dst[0] = *reinterpret_cast<const uint4*>(h16);
                dst[1] = *reinterpret_cast<const uint4*>(h16 + 8);
            }
            if (A.other) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float c = cs[i];
                    c += __shfl_xor_sync(0xffffffffu, c, 16);
                    c += __shfl_xor_sync(0xffffffffu, c, 8);
                    c += __shfl_xor_sync(0xffffffffu, c, 4);
                    c += __shfl_xor_sync(0xffffffffu, c, 2);
                    c += __shfl_xor_sync(0xffffffffu, c, 1);
                    cs[i] = c;
                }
                const int tc = t - lane;                    // first token of the chunk
                if (lane < 16 && tc < A.T) {
                    float mine = 0.f;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (i == lane) mine = cs[i];
                    A.colpart[(int64_t)(tc / 32) * A.r + kA + (lane >> 1) + 16 * (lane & 1)] = mine;
                }
            }
        }
    }

    // nothing reads or writes another CTA's shared memory after the second barrier
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512u);
    }
}

namespace {

template <int RB>
cudaError_t br_launch(const BrArgs& a, int T, cudaStream_t st) {
    constexpr int STAGE_B = BR_BK * RB * 2;
    constexpr int STAGE_X = BR_BK * 128 * 4;
    constexpr int STAGE_W = BR_BK * (RB / 32) * 4;
    constexpr int STAGE_G = BR_BK * 4;
    const int S = RB == 256 ? 3 : 4;
    const int red_bytes = 128 * (RB + 4) * 4;
    const int used = S * (STAGE_B + STAGE_X + STAGE_W + STAGE_G);
    const int ring = used > red_bytes ? used : red_bytes;
    // the sign words [K][r/32] as RB/32-word x 64-row boxes
    CUtensorMap bmap;
    if (!make_tensor_map_2d(&bmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, const_cast<uint32_t*>(a.bits), (uint64_t)a.r / 32,
                            (uint64_t)a.K, (uint64_t)a.r / 8, (uint32_t)(RB / 32), (uint32_t)BR_BK,
                            CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    // the activation [T][K] f32 as 32-column x 128-token boxes, 128-byte swizzle
    CUtensorMap xmap;
    if (!make_tensor_map_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, const_cast<float*>(a.act), (uint64_t)a.K,
                            (uint64_t)T, (uint64_t)a.K * 4, 32u, 128u, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const size_t smem = (size_t)ring + 16384 + sizeof(BrBars) + 1024;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int tiles = (T + 127) / 128, rbs = a.r / RB, nk = a.K / BR_BK;
    // K slices a cluster: the largest of 4, 2, 1 that keeps every CTA of the
    // grid resident at once and gives each slice at least two stages
    int CL = 4;
    while (CL > 1 && (CL * tiles * rbs > sms || nk < 2 * CL)) CL >>= 1;
    cudaError_t e = cudaFuncSetAttribute(blr_rank_kernel<RB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)CL, (unsigned)rbs, (unsigned)tiles);
    cfg.blockDim = dim3(BR_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)CL;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, blr_rank_kernel<RB>, xmap, bmap, a, S, CL);
}

}  // namespace

// res[t][k] = oscale * sum_j f16(act[t][j] * vec[j] * scale) * P[j][k] for the
// sign plane P of `bits` ([K][r/32]); st16 = f16(res * col * scale2) in the
// 32-group pair order; colpart[c][k] = sum over tokens 32c..32c+31 of
// res * other (if other).  Requirements: K % 64 == 0, r % 128 == 0, act and
// vec 16-byte aligned.
cudaError_t launch_blr_rank(const float* act, const float* vec, float scale, const uint32_t* bits, int T, int K,
                            int r, float oscale, float* res, const float* col, float scale2, uint16_t* st16,
                            const float* other, float* colpart, cudaStream_t st) {
    BrArgs a{act, vec, scale, bits, T, K, r, oscale, res, col, scale2, st16, other, colpart};
    if (r % 256 == 0) return br_launch<256>(a, T, st);
    return br_launch<128>(a, T, st);
}

}  // namespace tq2
