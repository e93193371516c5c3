// tq2_gemv.cu -- fused decode-shape GEMV for M <= 2 tokens.
//
//   out[m,n] = sum_k x[m,k] * W[n,k],  W[n,k] = (c-1)*d   (BlockTQ2_0_g128,
//   "oxibonsai-kernels 0.2.1, src/gpu_backend/metal_graph/tests_gemm_tq2.rs")
//
// One kernel per GEMV (no staging kernel, no scratch):
//   * A CTA owns 16 weight rows (one m16 fragment); its 8 warps split K.
//   * Before griddepcontrol.wait each lane loads the packed codes and scales
//     of its rows for its first K chunk: the weights never depend on earlier
//     work, so they stream in while the previous kernel on the stream drains.
//   * After the wait each warp converts the x values of its own K chunk to
//     the hi/lo f16 B fragments of mma.m16n8k16 (shared memory, warp-private)
//     together with the per-block correction sum_k (m_q + 1) x_k.
//   * Codes are decoded with decode_word_offset (shift + mask|magic, no
//     subtraction): the MMA accumulates (m_q + c) x per 128-block in f32; the
//     block result is d * (acc_hi + acc_lo - correction).
//   * The warps' partial sums meet in shared memory in a fixed order.
#include "ptx.cuh"
#include "tq2_internal.h"

namespace tq2 {

namespace {

constexpr int GV_WARPS = 8;
constexpr int GV_CHUNK = 4;            // 128-blocks per warp per chunk

__device__ __forceinline__ uint2 ldg_nc_u2(const uint8_t* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

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

template <int Q>
__device__ __forceinline__ uint32_t opair(uint32_t w) {
    if constexpr (Q == 0) return offset_pair<4>(w << 4);
    else if constexpr (Q == 1) return offset_pair<6>(w << 4);
    else if constexpr (Q == 2) return offset_pair<8>(w << 4);
    else if constexpr (Q == 3) return offset_pair<4>(w >> 2);
    else if constexpr (Q == 4) return offset_pair<6>(w >> 2);
    else if constexpr (Q == 5) return offset_pair<8>(w >> 2);
    else if constexpr (Q == 6) return offset_pair<4>(w >> 8);
    else return offset_pair<6>(w >> 8);
}

}  // namespace

// Shared memory per warp: xs[blk][step][col][t] (uint2 B fragments, col =
// 2*m + part) and corr[blk][m].
template <int MT>
struct GemvSmem {
    uint2 xs[GV_WARPS][GV_CHUNK][8][2 * MT][4];
    float corr[GV_WARPS][GV_CHUNK][MT];
    float red[GV_WARPS][16][MT];
};

template <int MT>
__global__ void __launch_bounds__(GV_WARPS * 32) tq2_gemv_kernel(const __grid_constant__ GemvTable tab) {
    __shared__ GemvSmem<MT> sm;
    // the job this CTA belongs to (jobs are laid out back to back in blockIdx.x)
    int job = 0;
    while (job + 1 < tab.njobs && (int)blockIdx.x >= tab.job[job + 1].cta0) ++job;
    const uint8_t* __restrict__ codes = tab.job[job].codes;
    const uint16_t* __restrict__ scales = tab.job[job].scales;
    const float* __restrict__ x = tab.job[job].x;
    float* __restrict__ out = tab.job[job].out;
    const int N = tab.job[job].N, K = tab.K;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int n0 = ((int)blockIdx.x - tab.job[job].cta0) * 16;
    const int nb = K >> 7;
    const int kb_begin = (nb * warp) / GV_WARPS, kb_end = (nb * (warp + 1)) / GV_WARPS;
    const int rowA = n0 + g, rowB = n0 + g + 8;
    const bool okA = rowA < N, okB = rowB < N;
    const int64_t pitch = K >> 2;
    const uint8_t* pA = codes + (int64_t)(okA ? rowA : 0) * pitch + 8 * t;
    const uint8_t* pB = codes + (int64_t)(okB ? rowB : 0) * pitch + 8 * t;
    const uint16_t* sA = scales + (int64_t)(okA ? rowA : 0) * nb;
    const uint16_t* sB = scales + (int64_t)(okB ? rowB : 0) * nb;

    // staging role of this lane: word (blk = lane/8, tq = (lane/2)%4, w = lane%2)
    const int st_blk = lane >> 3, st_t = (lane >> 1) & 3, st_w = lane & 1;

    float totA[MT], totB[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) totA[m] = totB[m] = 0.f;

    uint2 cA[GV_CHUNK], cB[GV_CHUNK];
    float dA[GV_CHUNK], dB[GV_CHUNK];
    auto load_chunk = [&](int kb0) {
#pragma unroll
        for (int c = 0; c < GV_CHUNK; ++c) {
            const int kb = kb0 + c;
            const bool v = kb < kb_end;
            cA[c] = (v && okA) ? ldg_nc_u2(pA + kb * 32) : make_uint2(0u, 0u);
            cB[c] = (v && okB) ? ldg_nc_u2(pB + kb * 32) : make_uint2(0u, 0u);
            dA[c] = (v && okA) ? __half2float(__ushort_as_half(__ldg(sA + kb))) : 0.f;
            dB[c] = (v && okB) ? __half2float(__ushort_as_half(__ldg(sB + kb))) : 0.f;
        }
    };
    load_chunk(kb_begin);
    pdl_wait();

#pragma unroll 1
    for (int kb0 = kb_begin; kb0 < kb_end; kb0 += GV_CHUNK) {
        // ---- stage this warp's x chunk: one 16-element word per lane and token
        {
            const int kb = kb0 + st_blk;
            const bool live = kb < kb_end;              // uniform within each 8-lane group
            const int k0 = (live ? kb : kb0) * 128 + 32 * st_t + 16 * st_w;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                float e[16];
                if (live) {
                    const float4* src = reinterpret_cast<const float4*>(x + (int64_t)m * K + k0);
                    const float4 q0 = __ldg(src), q1 = __ldg(src + 1), q2 = __ldg(src + 2), q3 = __ldg(src + 3);
                    e[0] = q0.x; e[1] = q0.y; e[2] = q0.z; e[3] = q0.w; e[4] = q1.x; e[5] = q1.y;
                    e[6] = q1.z; e[7] = q1.w; e[8] = q2.x; e[9] = q2.y; e[10] = q2.z; e[11] = q2.w;
                    e[12] = q3.x; e[13] = q3.y; e[14] = q3.z; e[15] = q3.w;
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) e[i] = 0.f;
                }
                float cs = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) cs = fmaf(offset_plus_one(i), e[i], cs);
                if (live) {
#pragma unroll
                    for (int sl = 0; sl < 4; ++sl) {         // k16 step 4*w + sl: pairs q = 2sl, 2sl+1
                        uint32_t h01, l01, h23, l23;
                        split2(e[2 * sl], e[2 * sl + 8], h01, l01);
                        split2(e[2 * sl + 1], e[2 * sl + 9], h23, l23);
                        const int s = 4 * st_w + sl;
                        sm.xs[warp][st_blk][s][2 * m][st_t] = make_uint2(h01, h23);
                        sm.xs[warp][st_blk][s][2 * m + 1][st_t] = make_uint2(l01, l23);
                    }
                }
                cs += __shfl_xor_sync(0xffffffffu, cs, 1);
                cs += __shfl_xor_sync(0xffffffffu, cs, 2);
                cs += __shfl_xor_sync(0xffffffffu, cs, 4);
                if (live && (lane & 7) == 0) sm.corr[warp][st_blk][m] = cs;
            }
            __syncwarp();
        }
        // ---- decode + MMA per block
#pragma unroll
        for (int c = 0; c < GV_CHUNK; ++c) {
            if (kb0 + c >= kb_end) break;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            const uint2* xb = &sm.xs[warp][c][0][0][0];
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t wa = (s < 4) ? cA[c].x : cA[c].y;
                const uint32_t wb = (s < 4) ? cB[c].x : cB[c].y;
                uint32_t a[4];
                switch (s & 3) {
                    case 0: a[0] = opair<0>(wa); a[1] = opair<0>(wb); a[2] = opair<1>(wa); a[3] = opair<1>(wb); break;
                    case 1: a[0] = opair<2>(wa); a[1] = opair<2>(wb); a[2] = opair<3>(wa); a[3] = opair<3>(wb); break;
                    case 2: a[0] = opair<4>(wa); a[1] = opair<4>(wb); a[2] = opair<5>(wa); a[3] = opair<5>(wb); break;
                    default: a[0] = opair<6>(wa); a[1] = opair<6>(wb); a[2] = opair<7>(wa); a[3] = opair<7>(wb); break;
                }
                uint2 b = make_uint2(0u, 0u);
                if (g < 2 * MT) b = xb[(s * 2 * MT + g) * 4 + t];
                mma_16816(acc, a, b.x, b.y, acc);
            }
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (t == m) {
                    const float corr = sm.corr[warp][c][m];
                    totA[m] = fmaf(dA[c], (acc[0] + acc[1]) - corr, totA[m]);
                    totB[m] = fmaf(dB[c], (acc[2] + acc[3]) - corr, totB[m]);
                }
        }
        __syncwarp();
        if (kb0 + GV_CHUNK < kb_end) load_chunk(kb0 + GV_CHUNK);
    }
    // The next kernel may start launching now: this CTA's loads are done, and
    // its prefetch cannot delay our (already finished) critical loads.
    pdl_launch_dependents();

#pragma unroll
    for (int m = 0; m < MT; ++m)
        if (t == m) {
            sm.red[warp][g][m] = totA[m];
            sm.red[warp][g + 8][m] = totB[m];
        }
    __syncthreads();
    if (threadIdx.x < 16 * MT) {
        const int m = threadIdx.x >> 4, r = threadIdx.x & 15;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < GV_WARPS; ++w) s += sm.red[w][r][m];
        if (n0 + r < N) out[(int64_t)m * N + n0 + r] = s;
    }
}

cudaError_t launch_gemv_table(const GemvTable& tab, int M, cudaStream_t st) {
    const int ctas = tab.job[tab.njobs - 1].cta0 + (tab.job[tab.njobs - 1].N + 15) / 16;
    const dim3 grid((unsigned)ctas), block(GV_WARPS * 32);
    if (M == 1) return launch_pdl(tq2_gemv_kernel<1>, grid, block, 0, st, tab);
    if (M == 2) return launch_pdl(tq2_gemv_kernel<2>, grid, block, 0, st, tab);
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemv(const uint8_t* codes, const uint16_t* scales, const float* x, float* out, int M, int N,
                        int K, cudaStream_t st) {
    GemvTable tab;
    tab.njobs = 1;
    tab.K = K;
    tab.job[0] = GemvJob{codes, scales, x, out, N, 0};
    return launch_gemv_table(tab, M, st);
}

}  // namespace tq2
