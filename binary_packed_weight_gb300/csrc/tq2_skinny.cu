// tq2_skinny.cu -- weight repack / unpack / dequant kernels and the skinny
// (M <= 16) ternary GEMM.
//
// Format: BlockTQ2_0_g128 ("oxibonsai-kernels 0.2.1, src/gpu_backend/
// metal_graph/tests_gemm_tq2.rs", test test_encode_gemm_tq2_matches_reference):
// per 128-wide block of a weight row, 32 bytes of 2-bit codes (element 4j+i at
// bits 2i of byte j) and an f16 scale d; W[n,k] = (c-1)*d.
//
// Device layout ("SoA"): codes uint8[N][K/4] (each row's qs bytes in K order),
// scales uint16[N][K/128] (f16 bits).
//
// Skinny GEMM: out[m,n] = sum_k x[m,k] W[n,k] for M <= 16 with f32
// activations.  The contraction runs on mma.sync m16n8k16 (f16 in, f32
// accumulate) because at M <= 16 the kernel is bound by issue slots: one
// HMMA replaces 2*M FFMAs per weight per thread.  Each x is carried as
// hi = f16(x) and lo = f16(x - hi) (two B columns); hi + lo differs from x by
// a relative residual of about 2^-22.  Weights enter the MMA as (c-1) in f16
// (exact); the block scale d multiplies the f32 block partial afterwards.
#include <mutex>

#include "../../include/tq2.h"
#include "ptx.cuh"
#include "tq2_internal.h"

namespace tq2 {

// --------------------------------------------------------------------------
// repack AoS (34-byte blocks) -> SoA planes, and back
// --------------------------------------------------------------------------
__global__ void repack_aos_kernel(const uint8_t* __restrict__ aos, uint8_t* __restrict__ codes,
                                  uint16_t* __restrict__ scales, int64_t nblocks) {
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;  // one byte of qs
    if (i >= nblocks * 32) return;
    const int64_t b = i >> 5;
    const int j = (int)(i & 31);
    const uint8_t* blk = aos + b * 34;
    codes[b * 32 + j] = blk[j];
    if (j == 0) scales[b] = (uint16_t)(blk[32] | ((uint16_t)blk[33] << 8));
}

__global__ void unpack_soa_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                                  uint8_t* __restrict__ aos, int64_t nblocks) {
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= nblocks * 32) return;
    const int64_t b = i >> 5;
    const int j = (int)(i & 31);
    uint8_t* blk = aos + b * 34;
    blk[j] = codes[b * 32 + j];
    if (j == 0) {
        const uint16_t d = scales[b];
        blk[32] = (uint8_t)(d & 0xFF);
        blk[33] = (uint8_t)(d >> 8);
    }
}

// Block-major copy of the scale plane for the tensor path: scales_t[b][n] =
// scales[n][b] for n < N, 0 for N <= n < Np.
__global__ void scales_t_kernel(const uint16_t* __restrict__ scales, uint16_t* __restrict__ scales_t, int64_t N,
                                int64_t nb, int64_t Np) {
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= nb * Np) return;
    const int64_t b = i / Np, n = i % Np;
    scales_t[i] = n < N ? scales[n * nb + b] : (uint16_t)0;
}

// Stage-tiled copy of the code plane for the tensor path: the 16 bytes (64
// codes) of row n in K-stage kc go to codes_t[n/128][kc][n%128], rows
// N <= n < Np zero.  One thread per 16-byte chunk, reading along a row.
__global__ void codes_t_kernel(const uint8_t* __restrict__ codes, uint8_t* __restrict__ codes_t, int64_t N,
                               int64_t nkc, int64_t Np) {
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= Np * nkc) return;
    const int64_t n = i / nkc, kc = i % nkc;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (n < N) v = *reinterpret_cast<const uint4*>(codes + (n * nkc + kc) * 16);
    *reinterpret_cast<uint4*>(codes_t + (((n >> 7) * nkc + kc) * 128 + (n & 127)) * 16) = v;
}

// W as f16 bits, natural order, through the same pair decode the GEMMs use:
// one thread per 32-bit code word (16 elements).
__global__ void dequant_f16_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                                   uint16_t* __restrict__ w, int64_t N, int64_t K) {
    const int64_t wi = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    const int64_t words_per_row = K / 16;
    if (wi >= N * words_per_row) return;
    const int64_t n = wi / words_per_row;
    const int64_t k0 = (wi % words_per_row) * 16;
    const uint32_t word = reinterpret_cast<const uint32_t*>(codes)[wi];
    const uint16_t dbits = scales[n * (K / 128) + k0 / 128];
    const __half2 d2 = __halves2half2(__ushort_as_half(dbits), __ushort_as_half(dbits));
    uint32_t p[8];
    decode_word(word, p);
    uint16_t* dst = w + n * K + k0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        __half2 v = __hmul2(*reinterpret_cast<__half2*>(&p[q]), d2);
        dst[q] = __half_as_ushort(__low2half(v));
        dst[q + 8] = __half_as_ushort(__high2half(v));
    }
}

// --------------------------------------------------------------------------
// skinny GEMM
// --------------------------------------------------------------------------
// Staged B fragments.  For n8 tile j, k16 step ks = 8*kb + s (kb: 128-block,
// s: step within the block) and lane (gq = lane/4, tq = lane%4) the uint2
// holds the two B registers of mma.m16n8k16: column gq is token 4j + gq/2,
// part gq%2 (0: hi, 1: lo); the K slots map to the A decode order:
//   b0,b1 = x[kbase + q], x[kbase + q + 8];  b2,b3 = x[kbase + q + 1], x[kbase + q + 9]
// with kbase = 128*kb + 32*tq + 16*(s/4) and q = 2*(s%4).
__device__ __forceinline__ uint16_t split_part(float v, int part) {
    const __half hi = __float2half_rn(v);
    if (part == 0) return __half_as_ushort(hi);
    return __half_as_ushort(__float2half_rn(v - __half2float(hi)));
}

__global__ void stage_x_frag_kernel(const float* __restrict__ x, uint2* __restrict__ xs, int M, int K,
                                    int ntiles) {
    pdl_wait();
    pdl_launch_dependents();
    const int KS = K >> 4;
    const int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (idx >= (int64_t)ntiles * KS * 32) return;
    const int lane = (int)(idx & 31);
    const int64_t rest = idx >> 5;
    const int ks = (int)(rest % KS);
    const int j = (int)(rest / KS);
    const int col = 8 * j + (lane >> 2);
    const int m = col >> 1, part = col & 1;
    if (m >= M) {
        xs[idx] = make_uint2(0u, 0u);
        return;
    }
    const int kb = ks >> 3, s = ks & 7;
    const int k = kb * 128 + 32 * (lane & 3) + 16 * (s >> 2) + 2 * (s & 3);
    const float* xr = x + (int64_t)m * K + k;
    const uint32_t b01 = (uint32_t)split_part(xr[0], part) | ((uint32_t)split_part(xr[8], part) << 16);
    const uint32_t b23 = (uint32_t)split_part(xr[1], part) | ((uint32_t)split_part(xr[9], part) << 16);
    xs[idx] = make_uint2(b01, b23);
}

// Pair q of a code word, q in 0..7 (elements q and q+8 of the word).
template <int Q>
__device__ __forceinline__ uint32_t pair_q(uint32_t w) {
    if constexpr (Q < 4) return decode_pair<2 * Q>(w);
    else return decode_pair<2 * (Q - 4)>(w >> 8);
}

__device__ __forceinline__ uint2 ldg_u2(const uint8_t* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// One CTA owns 16 weight rows (one m16 fragment); its W warps split the
// K blocks and reduce through shared memory.  Lane (g, t) of a warp reads
// bytes 8t..8t+7 of the 32-byte block of rows g and g+8: two code words per
// row per block, i.e. the 4 k16 steps s = 4*word + 0..3 of that word.
template <int NT>
__global__ void __launch_bounds__(256) tq2_skinny_kernel(const uint8_t* __restrict__ codes,
                                                         const uint16_t* __restrict__ scales,
                                                         const uint2* __restrict__ xs,
                                                         float* __restrict__ out, int M, int N, int K) {
    constexpr int CH = 4;                      // blocks loaded ahead per warp
    __shared__ float red[8][16][17];           // [warp][token][row]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = blockDim.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int n0 = blockIdx.x * 16;
    const int nb = K >> 7;
    const int KS = K >> 4;
    const int kb_begin = (nb * warp) / W, kb_end = (nb * (warp + 1)) / W;
    const int rowA = n0 + g, rowB = n0 + g + 8;
    const bool okA = rowA < N, okB = rowB < N;
    const int64_t pitch = K >> 2;
    const uint8_t* pA = codes + (int64_t)(okA ? rowA : 0) * pitch + 8 * t;
    const uint8_t* pB = codes + (int64_t)(okB ? rowB : 0) * pitch + 8 * t;
    const uint16_t* sA = scales + (int64_t)(okA ? rowA : 0) * nb;
    const uint16_t* sB = scales + (int64_t)(okB ? rowB : 0) * nb;

    pdl_launch_dependents();

    float tot[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) tot[j][i] = 0.f;

    bool waited = false;
#pragma unroll 1
    for (int kb0 = kb_begin; kb0 < kb_end; kb0 += CH) {
        uint2 cA[CH], cB[CH];
        float dA[CH], dB[CH];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int kb = kb0 + c;
            const bool v = kb < kb_end;
            cA[c] = (v && okA) ? ldg_u2(pA + kb * 32) : make_uint2(0u, 0u);
            cB[c] = (v && okB) ? ldg_u2(pB + kb * 32) : make_uint2(0u, 0u);
            dA[c] = (v && okA) ? __half2float(__ushort_as_half(__ldg(sA + kb))) : 0.f;
            dB[c] = (v && okB) ? __half2float(__ushort_as_half(__ldg(sB + kb))) : 0.f;
        }
        if (!waited) {           // the weights are immutable; x may come from the previous kernel
            pdl_wait();
            waited = true;
        }
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int kb = kb0 + c;
            if (kb >= kb_end) break;
            float acc[NT][4];
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;
            const uint2* xb = xs + ((int64_t)kb * 8) * 32 + lane;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t wa = (s < 4) ? cA[c].x : cA[c].y;
                const uint32_t wb = (s < 4) ? cB[c].x : cB[c].y;
                uint32_t a[4];
                switch (s & 3) {
                    case 0: a[0] = pair_q<0>(wa); a[1] = pair_q<0>(wb); a[2] = pair_q<1>(wa); a[3] = pair_q<1>(wb); break;
                    case 1: a[0] = pair_q<2>(wa); a[1] = pair_q<2>(wb); a[2] = pair_q<3>(wa); a[3] = pair_q<3>(wb); break;
                    case 2: a[0] = pair_q<4>(wa); a[1] = pair_q<4>(wb); a[2] = pair_q<5>(wa); a[3] = pair_q<5>(wb); break;
                    default: a[0] = pair_q<6>(wa); a[1] = pair_q<6>(wb); a[2] = pair_q<7>(wa); a[3] = pair_q<7>(wb); break;
                }
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const uint2 b = xb[((int64_t)j * KS + s) * 32];
                    mma_16816(acc[j], a, b.x, b.y, acc[j]);
                }
            }
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                tot[j][0] = fmaf(dA[c], acc[j][0], tot[j][0]);
                tot[j][1] = fmaf(dA[c], acc[j][1], tot[j][1]);
                tot[j][2] = fmaf(dB[c], acc[j][2], tot[j][2]);
                tot[j][3] = fmaf(dB[c], acc[j][3], tot[j][3]);
            }
        }
    }
    if (!waited) pdl_wait();

    // Columns 2t, 2t+1 of tile j are token 4j+t (hi, lo).
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int m = 4 * j + t;
        red[warp][m][g] = tot[j][0] + tot[j][1];
        red[warp][m][g + 8] = tot[j][2] + tot[j][3];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < M * 16; i += blockDim.x) {
        const int m = i >> 4, r = i & 15;
        float s = 0.f;
        for (int w = 0; w < W; ++w) s += red[w][m][r];
        if (n0 + r < N) out[(int64_t)m * N + n0 + r] = s;
    }
}

// --------------------------------------------------------------------------
// host launchers
// --------------------------------------------------------------------------
cudaError_t launch_repack(const uint8_t* aos_dev, uint8_t* codes, uint16_t* scales, int64_t nblocks,
                          cudaStream_t st) {
    const int64_t n = nblocks * 32;
    repack_aos_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(aos_dev, codes, scales, nblocks);
    return cudaGetLastError();
}

cudaError_t launch_scales_t(const uint16_t* scales, uint16_t* scales_t, int64_t N, int64_t nb, int64_t Np,
                            cudaStream_t st) {
    const int64_t n = nb * Np;
    scales_t_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(scales, scales_t, N, nb, Np);
    return cudaGetLastError();
}

cudaError_t launch_codes_t(const uint8_t* codes, uint8_t* codes_t, int64_t N, int64_t K, int64_t Np,
                           cudaStream_t st) {
    const int64_t n = Np * (K / 64);
    codes_t_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(codes, codes_t, N, K / 64, Np);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t* codes, const uint16_t* scales, uint8_t* aos_dev, int64_t nblocks,
                          cudaStream_t st) {
    const int64_t n = nblocks * 32;
    unpack_soa_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(codes, scales, aos_dev, nblocks);
    return cudaGetLastError();
}

cudaError_t launch_dequant_f16(const uint8_t* codes, const uint16_t* scales, uint16_t* w, int64_t N, int64_t K,
                               cudaStream_t st) {
    const int64_t n = N * (K / 16);
    dequant_f16_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(codes, scales, w, N, K);
    return cudaGetLastError();
}

size_t skinny_scratch_bytes(int64_t M, int64_t K) {
    const int64_t ntiles = (M + 3) / 4;
    return (size_t)(ntiles * (K / 16) * 32) * sizeof(uint2);
}

cudaError_t launch_skinny(const uint8_t* codes, const uint16_t* scales, const float* x, float* out, int M,
                          int N, int K, void* scratch, cudaStream_t st) {
    const int ntiles = (M + 3) / 4;
    uint2* xs = reinterpret_cast<uint2*>(scratch);
    const int64_t nthr = (int64_t)ntiles * (K / 16) * 32;
    cudaError_t e = launch_pdl(stage_x_frag_kernel, dim3((unsigned)((nthr + 255) / 256)), dim3(256), 0, st,
                               x, xs, M, K, ntiles);
    if (e != cudaSuccess) return e;
    const int nb = K / 128;
    const int W = nb < 8 ? nb : 8;
    const dim3 grid((unsigned)((N + 15) / 16)), block((unsigned)(32 * W));
    const uint2* cxs = xs;
    switch (ntiles) {
        case 1: return launch_pdl(tq2_skinny_kernel<1>, grid, block, 0, st, codes, scales, cxs, out, M, N, K);
        case 2: return launch_pdl(tq2_skinny_kernel<2>, grid, block, 0, st, codes, scales, cxs, out, M, N, K);
        case 3: return launch_pdl(tq2_skinny_kernel<3>, grid, block, 0, st, codes, scales, cxs, out, M, N, K);
        case 4: return launch_pdl(tq2_skinny_kernel<4>, grid, block, 0, st, codes, scales, cxs, out, M, N, K);
        default: return cudaErrorInvalidValue;
    }
}

unsigned int read_clear_dev_error_skinny(cudaStream_t st) {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_dev_error, sizeof(v), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return 0;
    cudaMemcpyToSymbolAsync(g_dev_error, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
    cudaStreamSynchronize(st);
    return v;
}

}  // namespace tq2

// --------------------------------------------------------------------------
// Allocation-free variant of the skinny GEMM.
//
// Some callers must not allocate device memory while they run a GEMM: a
// plugin or custom-op interface that forbids allocation inside its enqueue
// call, a serving process that reserved all device memory up front, or a
// real-time loop where an allocator call could stall or fail.  For them,
// tq2_gemm_skinny_static runs the fused GEMV where it applies (it has no
// scratch) and otherwise keeps the staged kernel's scratch (the hi/lo f16
// fragments of x) in the fixed device array below instead of asking the
// stream-ordered allocator; it calls no allocating routine at all.
// --------------------------------------------------------------------------
namespace {

constexpr size_t kStaticScratchBytes = size_t(1) << 20;     // 1 MiB per device
// Lives in every GPU that loads this library until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void* g_static_scratch_ptr[kMaxDevices] = {};
std::mutex g_static_scratch_mutex;

// Device address of g_static_scratch on the current device, looked up once
// per device (host code only sees a stand-in for the array, never its device
// address, so the address must come from cudaGetSymbolAddress).  The cache
// assumes that the device's primary context lives as long as the process:
// after cudaDeviceReset the cached address is stale, so a process that resets
// a device must not call tq2_gemm_skinny_static on it again.
cudaError_t static_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_static_scratch_mutex);
    if (!g_static_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        g_static_scratch_ptr[dev] = p;
    }
    *out = g_static_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" TQ2_API tq2_status tq2_gemm_skinny_static(tq2_handle h, const float* x, float* out, int64_t M,
                                                     int64_t N, int64_t K, void* stream) {
    if (!h) return (tq2_status)tq2::set_error(TQ2_EINVAL, "tq2_gemm_skinny_static: null handle");
    if (M == 0) return TQ2_OK;
    if (!x || !out) return (tq2_status)tq2::set_error(TQ2_EINVAL, "tq2_gemm_skinny_static: null pointer");
    if (M < 0 || M > 16)
        return (tq2_status)tq2::set_error(TQ2_ESHAPE, "tq2_gemm_skinny_static: need 1 <= M <= 16 (M=%lld)", (long long)M);
    if (N != h->N || K != h->K)
        return (tq2_status)tq2::set_error(TQ2_ESHAPE, "tq2_gemm_skinny_static: (N,K)=(%lld,%lld) but the handle holds (%lld,%lld)",
                                     (long long)N, (long long)K, (long long)h->N, (long long)h->K);
    if ((reinterpret_cast<uintptr_t>(x) & 15) != 0)
        return (tq2_status)tq2::set_error(TQ2_EINVAL, "tq2_gemm_skinny_static: x must be 16-byte aligned");
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device)
        return (tq2_status)tq2::set_error(TQ2_EINVAL,
                                          "tq2_gemm_skinny_static: the handle lives on device %d but device %d is "
                                          "current (the fixed scratch array is per device)",
                                          h->device, dev);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // Shapes the fused GEMV takes need no scratch at all: the same kernel as
    // tq2_gemm, so the results are the same bit for bit.
    if (tq2::gemv_supports((int)M, K)) {
        cudaError_t e = tq2::launch_gemv(&h, &x, &out, 1, (int)M, st);
        if (e != cudaSuccess)
            return (tq2_status)tq2::set_error(TQ2_ECUDA, "tq2_gemm_skinny_static: gemv launch: %s", cudaGetErrorString(e));
        return TQ2_OK;
    }
    const size_t need = tq2::skinny_scratch_bytes(M, K);
    if (need > kStaticScratchBytes)
        return (tq2_status)tq2::set_error(TQ2_ESHAPE,
                                     "tq2_gemm_skinny_static: needs %zu bytes of scratch for M=%lld K=%lld, above the "
                                     "fixed %zu-byte area (ceil(M/4)*K*16 must be <= %zu)",
                                     need, (long long)M, (long long)K, kStaticScratchBytes, kStaticScratchBytes);
    void* scratch = nullptr;
    cudaError_t e = static_scratch(&scratch);
    if (e != cudaSuccess)
        return (tq2_status)tq2::set_error(TQ2_ECUDA, "tq2_gemm_skinny_static: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    // Every element of the scratch that the GEMM reads is written first by the
    // staging kernel of the same call, so nothing needs clearing.
    e = tq2::launch_skinny(h->codes, h->scales, x, out, (int)M, (int)N, (int)K, scratch, st);
    if (e != cudaSuccess)
        return (tq2_status)tq2::set_error(TQ2_ECUDA, "tq2_gemm_skinny_static: launch: %s", cudaGetErrorString(e));
    return TQ2_OK;
}

// --------------------------------------------------------------------------
// Test export: a bounded device-side wait that runs out.
//
// Every wait inside the library's kernels gives up after a bounded time,
// records the timeout in the device error word and returns, so that a lost
// hand-off ends as a status (tq2_device_status -> TQ2_ETIMEOUT) instead of a
// hung GPU.  This kernel exercises that path on purpose and nothing else:
// one thread initialises a shared-memory mbarrier that expects one arrival,
// never arrives on it, waits for its first phase with a bound of limit_ns,
// records the timeout and returns.  It touches no other memory.
// --------------------------------------------------------------------------
namespace tq2 {
namespace {

__global__ void wait_runs_out_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait_sleep(&bar, 0u, 1000u)) {       // phase 0 never completes
        if (global_timer_ns() - t0 > limit_ns) {
            record_timeout();
            return;
        }
    }
}

}  // namespace
}  // namespace tq2

extern "C" TQ2_API tq2_status tq2_debug_wait_timeout(uint64_t limit_ns, void* stream) {
    if (limit_ns == 0 || limit_ns > tq2::WAIT_LIMIT_NS)
        return (tq2_status)tq2::set_error(TQ2_EINVAL, "tq2_debug_wait_timeout: need 0 < limit_ns <= %llu",
                                          (unsigned long long)tq2::WAIT_LIMIT_NS);
    tq2::wait_runs_out_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return (tq2_status)tq2::set_error(TQ2_ECUDA, "tq2_debug_wait_timeout: launch: %s", cudaGetErrorString(e));
    return TQ2_OK;
}
