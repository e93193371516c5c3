// umma_core.cuh -- the tcgen05 GEMM core shared by the ternary TQ2 path and
// the binary low-rank (blr) layer:
//
//   D[t, n] = sum_k act[t, k] * P[n, k]
//
// P is a packed plane (2-bit ternary codes with f16 block scales, or 1-bit
// signs) decoded on chip; act is an f16 activation matrix staged in the K
// order the decoder emits pairs in.  One CTA computes a 128 (plane rows) x BN
// (tokens) tile:
//   * four decoder warps (one plane row per thread = its TMEM lane) write the
//     decoded f16 pairs into tensor memory with tcgen05.st: the MMA's A
//     operand never passes through shared memory;
//   * one thread issues TMA loads of the activation tile (B operand, 128-byte
//     swizzle) into a 4-stage shared-memory ring;
//   * one thread issues tcgen05.mma (kind::f16, f32 accumulate in TMEM) and
//     frees stages with tcgen05.commit;
//   * the decoder warps then read the accumulator (tcgen05.ld) and run the
//     epilogue policy of the call.
// All waits are bounded (mbar_wait); a timeout records an error and drains.
#pragma once

#include "ptx.cuh"
#include "tq2_internal.h"

namespace tq2 {

constexpr int UM_BM = 128;       // plane rows per CTA = MMA M
constexpr int UM_BK = 64;        // K per pipeline stage (128 bytes of f16)
constexpr int UM_STAGES = 4;
constexpr int UM_THREADS = 256;  // warp 0 TMA, warp 1 MMA, warp 2 TMEM, warps 4-7 decode + epilogue

struct UmmaBars {
    uint64_t full_b[UM_STAGES];
    uint64_t full_a[UM_STAGES];
    uint64_t empty[UM_STAGES];
    uint64_t done;
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
// A decoder turns plane row `row` (valid iff ok) of K-stage i (64 elements)
// into 32 f16 pairs v[0..31]; column j of the stage holds K positions 2j,2j+1
// of the permuted order the activations are staged in.

// TQ2 codes: 16 bytes of codes per stage, element e of a 16-element word at
// bits 2e; pair q = (element q, element q+8); the block scale is folded in:
// (c-1)*d is exact in f16.  Activations staged with 16-element groups.
struct DecTQ2 {
    const uint8_t* codes;      // [rows][K/4]
    const uint16_t* scales;    // [rows][K/128]
    int64_t pitch;             // K/4
    int nb;                    // K/128
    struct Raw { uint4 c; uint16_t d; };
    __device__ __forceinline__ Raw load(int row, bool ok, int kc) const {
        Raw r;
        if (ok) {
            r.c = ldg_u4_nc(codes + (int64_t)row * pitch + (int64_t)kc * 16);
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
                __half2 h = __hmul2(*reinterpret_cast<__half2*>(&p[q]), d2);
                v[w * 8 + q] = *reinterpret_cast<uint32_t*>(&h);
            }
        }
    }
};

// Sign bits: 2 words of 32 signs per stage (bit b of word w = element 32w+b,
// set = +1); pair p = (element p, element p+16) of a word.  Activations
// staged with 32-element groups.
struct DecSign {
    const uint32_t* bits;      // [rows][K/32]
    int64_t words;             // K/32
    struct Raw { uint2 w; };
    __device__ __forceinline__ Raw load(int row, bool ok, int kc) const {
        Raw r;
        r.w = ok ? ldg_u2_nc(bits + (int64_t)row * words + (int64_t)kc * 2) : make_uint2(0u, 0u);
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

// --------------------------------------------------------------- epilogues ----
enum EpiMode : int {
    EPI_STORE = 0,        // out[t][n] = acc * oscale
    EPI_ATOMIC = 1,       // out[t][n] += acc * oscale (atomic; two K splits at most)
    EPI_PARTIAL = 2,      // out[z][t][n] = acc (split-K partial, z = blockIdx.z)
    EPI_SCALE = 3,        // out[t][n] = acc * oscale * vec[n]; out2[t][n] = acc * oscale if out2
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
};

// ----------------------------------------------------------------- kernel ----
template <class Dec, int MODE>
__global__ void __launch_bounds__(UM_THREADS, 1)
umma_gemm_kernel(const __grid_constant__ CUtensorMap xmap, const Dec dec, const EpiArgs ep, int T, int R, int K,
                 int BN, int tmem_cols) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int stage_bytes = BN * 128;
    UmmaBars* bars = reinterpret_cast<UmmaBars*>(smem + UM_STAGES * stage_bytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * UM_BM;
    const int m0 = blockIdx.y * BN;
    const int nk_total = K / UM_BK;
    const int kc0 = (int)(((int64_t)nk_total * blockIdx.z) / gridDim.z);
    const int kc1 = (int)(((int64_t)nk_total * (blockIdx.z + 1)) / gridDim.z);
    const int nk = kc1 - kc0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < UM_STAGES; ++s) {
            mbar_init(&bars->full_b[s], 1);
            mbar_init(&bars->full_a[s], 4);
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->done, 1);
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
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t a_col0 = (uint32_t)BN;
    volatile int* abort_flag = &bars->abort;

    pdl_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {                       // TMA producer (activation tiles)
            pdl_wait();
            int issued = 0;
            for (int i = 0; i < nk; ++i) {
                const int s = i % UM_STAGES;
                const uint32_t ph = (uint32_t)(i / UM_STAGES) & 1u;
                if (i >= UM_STAGES && !mbar_wait(&bars->empty[s], ph ^ 1u)) { *abort_flag = 1; break; }
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&bars->full_b[s], (uint32_t)stage_bytes);
                tma_load_2d(smem + s * stage_bytes, &xmap, &bars->full_b[s], (kc0 + i) * UM_BK, m0);
                ++issued;
            }
            if (*abort_flag) {                 // let copies already issued land before exit
                for (int i = issued - UM_STAGES < 0 ? 0 : issued - UM_STAGES; i < issued; ++i)
                    mbar_wait(&bars->full_b[i % UM_STAGES], (uint32_t)(i / UM_STAGES) & 1u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {                       // MMA issuer
            const uint32_t idesc = idesc_f16_f32(UM_BM, (uint32_t)BN);
            for (int i = 0; i < nk; ++i) {
                const int s = i % UM_STAGES;
                const uint32_t ph = (uint32_t)(i / UM_STAGES) & 1u;
                if (!mbar_wait(&bars->full_b[s], ph) || !mbar_wait(&bars->full_a[s], ph) || *abort_flag) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(smem + s * stage_bytes));
#pragma unroll
                for (int j = 0; j < UM_BK / 16; ++j)
                    umma_f16_ts(tmem, tmem + a_col0 + (uint32_t)(s * (UM_BK / 2) + j * 8), bdesc + (uint64_t)(2 * j),
                                idesc, (i > 0 || j > 0) ? 1u : 0u);
                umma_commit(&bars->empty[s]);
            }
            umma_commit(&bars->done);
        }
    } else if (warp >= 4) {
        const int q = warp & 3;
        const int row = n0 + q * 32 + lane;
        const bool rok = row < R;
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);

        auto process = [&](int i, const typename Dec::Raw& raw) -> bool {
            const int s = i % UM_STAGES;
            const uint32_t ph = (uint32_t)(i / UM_STAGES) & 1u;
            if (i >= UM_STAGES && !mbar_wait(&bars->empty[s], ph ^ 1u)) return false;
            if (*abort_flag) return false;
            tc_fence_after();
            uint32_t v[32];
            dec.decode(raw, v);
            tmem_st_32x32b_x32(lane_addr + a_col0 + (uint32_t)(s * (UM_BK / 2)), v);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->full_a[s]);
            return true;
        };
        auto ld = [&](int i) { return dec.load(rok ? row : 0, rok && i < nk, kc0 + (i < nk ? i : 0)); };

        typename Dec::Raw r0 = ld(0), r1 = ld(1), r2 = ld(2), r3 = ld(3);
        bool ok = true;
        for (int i = 0; i < nk && ok; i += 4) {
            ok = process(i, r0);
            r0 = ld(i + 4);
            if (ok && i + 1 < nk) { ok = process(i + 1, r1); r1 = ld(i + 5); }
            if (ok && i + 2 < nk) { ok = process(i + 2, r2); r2 = ld(i + 6); }
            if (ok && i + 3 < nk) { ok = process(i + 3, r3); r3 = ld(i + 7); }
        }
        if (!ok) *abort_flag = 1;

        // ---------------- epilogue ----------------
        if (mbar_wait(&bars->done, 0) && !*abort_flag) {
            tc_fence_after();
            pdl_wait();
            float colacc = 0.f;
            for (int cc = 0; cc < BN; cc += 32) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(lane_addr + (uint32_t)cc, v);
                tmem_wait_ld();
                if (!rok) continue;
                const float vs = (MODE == EPI_SCALE || MODE == EPI_SCALE_COLSUM) ? ep.vec[row] : 1.f;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int m = m0 + cc + i;
                    if (m >= T) break;
                    const float a = __uint_as_float(v[i]);
                    const int64_t o = (int64_t)m * ep.ldo + row;
                    if (MODE == EPI_STORE) {
                        ep.out[o] = a * ep.oscale;
                    } else if (MODE == EPI_ATOMIC) {
                        atomicAdd(ep.out + o, a * ep.oscale);
                    } else if (MODE == EPI_PARTIAL) {
                        ep.out[(int64_t)blockIdx.z * T * ep.ldo + o] = a;
                    } else {
                        const float w = a * ep.oscale;
                        if (MODE == EPI_SCALE || MODE == EPI_SCALE_COLSUM) {
                            ep.out[o] = w * vs;
                            if (MODE == EPI_SCALE && ep.out2) ep.out2[o] = w;
                        }
                        if (MODE == EPI_SCALE_COLSUM || MODE == EPI_COLSUM) colacc = fmaf(w, ep.other[o], colacc);
                    }
                }
            }
            if ((MODE == EPI_SCALE_COLSUM || MODE == EPI_COLSUM) && rok)
                ep.colpart[(int64_t)blockIdx.y * ep.ldo + row] = colacc;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)tmem_cols);
    }
}

// Host: launch one GEMM.  act16 is f16 [T][K] (row pitch K), staged in the
// decoder's K order; R = plane rows; splits = K splits (gridDim.z).
template <class Dec, int MODE>
cudaError_t launch_umma(const Dec& dec, const EpiArgs& ep, const void* act16, int T, int R, int K, int BN, int splits,
                        cudaStream_t st) {
    CUtensorMap xmap;
    if (!make_tensor_map_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, const_cast<void*>(act16), (uint64_t)K,
                            (uint64_t)T, (uint64_t)K * 2, UM_BK, (uint32_t)BN, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    int tmem_cols = 32;
    while (tmem_cols < BN + UM_STAGES * (UM_BK / 2)) tmem_cols <<= 1;
    const size_t smem = (size_t)UM_STAGES * BN * 128 + sizeof(UmmaBars) + 1024;
    const dim3 grid((unsigned)((R + UM_BM - 1) / UM_BM), (unsigned)((T + BN - 1) / BN), (unsigned)splits);
    cudaError_t e = cudaFuncSetAttribute(umma_gemm_kernel<Dec, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(umma_gemm_kernel<Dec, MODE>, grid, dim3(UM_THREADS), smem, st, xmap, dec, ep, T, R, K, BN,
                      tmem_cols);
}

inline int umma_pick_bn(int T) {
    if (T >= 256) return 256;
    return ((T + 31) / 32) * 32;
}

}  // namespace tq2
