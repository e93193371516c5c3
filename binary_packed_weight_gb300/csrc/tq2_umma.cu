// tq2_umma.cu -- large-M ternary GEMM on the 5th-generation tensor cores.
//
//   out[m,n] = sum_k x[m,k] * W[n,k],   W[n,k] = (c-1)*d   (BlockTQ2_0_g128,
//   "oxibonsai-kernels 0.2.1, src/gpu_backend/metal_graph/tests_gemm_tq2.rs")
//
// Activations are staged once to f16 (round to nearest even); the weights are
// expanded on chip to (c-1)*d in f16, which is exact (the v10 parity test on
// that page relies on the same fact), so the block scale needs no epilogue.
//
// One CTA computes a 128 (weight rows) x BN (tokens) tile of out^T:
//   * the MMA's A operand is the decoded weight tile, written straight into
//     tensor memory by four decoder warps (one weight row per thread, so a
//     thread's row is its TMEM lane) -- no shared-memory traffic for A;
//   * the B operand is the f16 activation tile, loaded by TMA with 128-byte
//     swizzling into a 4-stage shared-memory ring;
//   * one elected thread issues tcgen05.mma (kind::f16, f32 accumulate) into
//     a TMEM accumulator of BN columns and commits each stage back to the
//     producers through mbarriers;
//   * the decoder warps then read the accumulator with tcgen05.ld and store
//     out[m][n] (a warp writes 32 consecutive n of one token: 128 bytes).
// The K order inside every 16-element group is permuted the same way on both
// operands: position 2q holds element q and 2q+1 holds element q+8, which is
// the order in which two-code pairs fall out of a 32-bit code word.
#include "ptx.cuh"
#include "tq2_internal.h"

namespace tq2 {

constexpr int UM_BM = 128;       // weight rows per CTA = MMA M
constexpr int UM_BK = 64;        // K elements per pipeline stage (128 bytes of f16)
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

__device__ __forceinline__ uint4 ldg_u4_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// x f32 [M][K] -> f16 [M][K] in the permuted 16-group order; optionally
// zero `zero_out` (split-K accumulation target).
__global__ void stage_x_f16_kernel(const float* __restrict__ x, uint32_t* __restrict__ xh, int64_t M,
                                   int64_t K, float* __restrict__ zero_out, int64_t zero_n) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    const int64_t groups = M * (K / 16);
    for (int64_t gi = tid; gi < groups; gi += nthreads) {
        const float4* src = reinterpret_cast<const float4*>(x + gi * 16);
        const float4 a = src[0], b = src[1], c = src[2], d = src[3];
        const float lo[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        const float hi[8] = {c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
        uint32_t o[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const __half2 h = __floats2half2_rn(lo[q], hi[q]);   // .x = element q, .y = element q+8
            o[q] = *reinterpret_cast<const uint32_t*>(&h);
        }
        uint4* dst = reinterpret_cast<uint4*>(xh + gi * 8);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
    for (int64_t i = tid; i < zero_n; i += nthreads) zero_out[i] = 0.f;
}

template <bool ATOMIC>
__global__ void __launch_bounds__(UM_THREADS, 1)
tq2_umma_kernel(const __grid_constant__ CUtensorMap xmap, const uint8_t* __restrict__ codes,
                const uint16_t* __restrict__ scales, float* __restrict__ out, int M, int N, int K, int BN,
                int tmem_cols) {
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
    const uint32_t a_col0 = (uint32_t)BN;        // A stages follow the BN accumulator columns
    volatile int* abort_flag = &bars->abort;

    pdl_launch_dependents();

    if (warp == 0) {
        // ---------------- TMA producer: activation tiles ----------------
        if (lane == 0) {
            pdl_wait();
            for (int i = 0; i < nk; ++i) {
                const int s = i % UM_STAGES;
                const uint32_t ph = (uint32_t)(i / UM_STAGES) & 1u;
                if (i >= UM_STAGES && !mbar_wait(&bars->empty[s], ph ^ 1u)) { *abort_flag = 1; break; }
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&bars->full_b[s], (uint32_t)stage_bytes);
                tma_load_2d(smem + s * stage_bytes, &xmap, &bars->full_b[s], (kc0 + i) * UM_BK, m0);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(UM_BM, (uint32_t)BN);
            bool ok = true;
            for (int i = 0; i < nk && ok; ++i) {
                const int s = i % UM_STAGES;
                const uint32_t ph = (uint32_t)(i / UM_STAGES) & 1u;
                if (!mbar_wait(&bars->full_b[s], ph) || !mbar_wait(&bars->full_a[s], ph) || *abort_flag) {
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(smem + s * stage_bytes));
#pragma unroll
                for (int j = 0; j < UM_BK / 16; ++j)
                    umma_f16_ts(tmem, tmem + a_col0 + (uint32_t)(s * (UM_BK / 2) + j * 8),
                                bdesc + (uint64_t)(2 * j), idesc, (i > 0 || j > 0) ? 1u : 0u);
                umma_commit(&bars->empty[s]);
            }
            umma_commit(&bars->done);
        }
    } else if (warp >= 4) {
        // ---------------- decoders (one weight row per thread) ----------------
        const int q = warp & 3;
        const int row = n0 + q * 32 + lane;
        const bool rok = row < N;
        const int64_t pitch = K / 4;
        const uint8_t* cp = codes + (int64_t)(rok ? row : 0) * pitch + (int64_t)kc0 * 16;
        const uint16_t* sp = scales + (int64_t)(rok ? row : 0) * (K / 128);
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);

        auto load = [&](int i, uint4& c, uint16_t& d) {
            if (rok && i < nk) {
                c = ldg_u4_stream(cp + (int64_t)i * 16);
                d = __ldg(sp + (kc0 + i) / 2);
            } else {
                c = make_uint4(0u, 0u, 0u, 0u);
                d = 0;
            }
        };
        auto process = [&](int i, const uint4& c, uint16_t dbits) -> bool {
            const int s = i % UM_STAGES;
            const uint32_t ph = (uint32_t)(i / UM_STAGES) & 1u;
            if (i >= UM_STAGES && !mbar_wait(&bars->empty[s], ph ^ 1u)) return false;
            if (*abort_flag) return false;
            tc_fence_after();
            const __half2 d2 = __halves2half2(__ushort_as_half(dbits), __ushort_as_half(dbits));
            uint32_t v[32];
            uint32_t p[8];
            const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                decode_word(words[w], p);
#pragma unroll
                for (int qq = 0; qq < 8; ++qq) {
                    __half2 h = __hmul2(*reinterpret_cast<__half2*>(&p[qq]), d2);
                    v[w * 8 + qq] = *reinterpret_cast<uint32_t*>(&h);
                }
            }
            tmem_st_32x32b_x32(lane_addr + a_col0 + (uint32_t)(s * (UM_BK / 2)), v);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->full_a[s]);
            return true;
        };

        uint4 c0, c1, c2, c3;
        uint16_t d0, d1, d2, d3;
        load(0, c0, d0);
        load(1, c1, d1);
        load(2, c2, d2);
        load(3, c3, d3);
        bool ok = true;
        for (int i = 0; i < nk && ok; i += 4) {
            ok = process(i, c0, d0);
            load(i + 4, c0, d0);
            if (ok && i + 1 < nk) { ok = process(i + 1, c1, d1); load(i + 5, c1, d1); }
            if (ok && i + 2 < nk) { ok = process(i + 2, c2, d2); load(i + 6, c2, d2); }
            if (ok && i + 3 < nk) { ok = process(i + 3, c3, d3); load(i + 7, c3, d3); }
        }
        if (!ok) *abort_flag = 1;

        // ---------------- epilogue ----------------
        if (mbar_wait(&bars->done, 0) && !*abort_flag) {
            tc_fence_after();
            pdl_wait();
            for (int cc = 0; cc < BN; cc += 32) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(lane_addr + (uint32_t)cc, v);
                tmem_wait_ld();
                if (rok) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int m = m0 + cc + i;
                        if (m < M) {
                            float* o = out + (int64_t)m * N + row;
                            if (ATOMIC) atomicAdd(o, __uint_as_float(v[i]));
                            else *o = __uint_as_float(v[i]);
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)tmem_cols);
    }
}

// --------------------------------------------------------------------------
size_t tensor_scratch_bytes(int64_t M, int64_t K) { return (size_t)(M * K * 2); }

static int pick_bn(int M) {
    if (M >= 256) return 256;
    return ((M + 31) / 32) * 32;
}

cudaError_t launch_tensor(const tq2_weight* w, const float* x, float* out, int M, void* scratch,
                          cudaStream_t st) {
    const int N = (int)w->N, K = (int)w->K;
    const int BN = pick_bn(M);
    const int tiles_n = (N + UM_BM - 1) / UM_BM;
    const int tiles_m = (M + BN - 1) / BN;
    const int nk = K / UM_BK;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int splits = (tiles_n * tiles_m * 4 < sms * 3 && nk >= 4) ? 2 : 1;

    uint32_t* xh = reinterpret_cast<uint32_t*>(scratch);
    const int64_t groups = (int64_t)M * (K / 16);
    int64_t blocks = (groups + 255) / 256;
    if (blocks > 4 * (int64_t)sms * 8) blocks = 4 * (int64_t)sms * 8;
    if (blocks < 1) blocks = 1;
    cudaError_t e = launch_pdl(stage_x_f16_kernel, dim3((unsigned)blocks), dim3(256), 0, st, x, xh, (int64_t)M,
                               (int64_t)K, out, splits > 1 ? (int64_t)M * N : (int64_t)0);
    if (e != cudaSuccess) return e;

    CUtensorMap xmap;
    if (!make_tensor_map_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xh, (uint64_t)K, (uint64_t)M,
                            (uint64_t)K * 2, UM_BK, (uint32_t)BN, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;

    int tmem_cols = 32;
    while (tmem_cols < BN + UM_STAGES * (UM_BK / 2)) tmem_cols <<= 1;
    const size_t smem = (size_t)UM_STAGES * BN * 128 + sizeof(UmmaBars) + 1024;
    const dim3 grid((unsigned)tiles_n, (unsigned)tiles_m, (unsigned)splits);
    if (splits > 1) {
        cudaFuncSetAttribute(tq2_umma_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        return launch_pdl(tq2_umma_kernel<true>, grid, dim3(UM_THREADS), smem, st, xmap, w->codes, w->scales,
                          out, M, N, K, BN, tmem_cols);
    }
    cudaFuncSetAttribute(tq2_umma_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return launch_pdl(tq2_umma_kernel<false>, grid, dim3(UM_THREADS), smem, st, xmap, w->codes, w->scales, out,
                      M, N, K, BN, tmem_cols);
}

unsigned int read_clear_dev_error_umma(cudaStream_t st) {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_dev_error, sizeof(v), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return 0;
    cudaMemcpyToSymbolAsync(g_dev_error, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
    cudaStreamSynchronize(st);
    return v;
}

}  // namespace tq2
