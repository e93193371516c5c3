// tq2_umma.cu -- large-M ternary GEMM on the 5th-generation tensor cores.
//
//   out[m,n] = sum_k x[m,k] * W[n,k],   W[n,k] = (c-1)*d   (BlockTQ2_0_g128,
//   "oxibonsai-kernels 0.2.1, src/gpu_backend/metal_graph/tests_gemm_tq2.rs")
//
// Activations are staged once to f16 (round to nearest even); the weights are
// expanded on chip to (c-1)*d in f16, which is exact (the v10 parity test on
// that page relies on the same fact), so the block scale needs no epilogue.
//
// The GEMM runs on the persistent tcgen05 core (umma_core.cuh) with the TQ2
// decoder: a CTA computes 128 weight rows x BN tokens of out^T; TMA streams
// the 2-bit code tiles and block scales into a deep shared-memory ring and
// the f16 activation tiles into another; decoder warps expand the codes into
// the f16 A operand (tensor memory for BN <= 128, else a swizzled
// shared-memory ring); one warp issues the MMAs into two tensor-memory
// accumulators, and four epilogue warps store out[m][n] while the next
// tile's MMAs run.
// The K order inside every 16-element group is permuted the same way on both
// operands: position 2q holds element q and 2q+1 holds element q+8, which is
// the order in which two-code pairs fall out of a 32-bit code word.
#include "tq2_internal.h"
#include "umma_core.cuh"

namespace tq2 {

// x f32 [M][K] -> f16 [M][K] in the permuted 16-group order (position 2q =
// element q, 2q+1 = element q+8, the pair order of a 32-bit code word);
// optionally zero `zero_out` (split-K accumulation target).
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

size_t tensor_scratch_bytes(int64_t M, int64_t K) { return (size_t)(M * K * 2); }

bool make_umma_maps(tq2_weight* w) {
    return plane_maps_tq2(w->umma_maps, w->codes_t, w->scales_t, (int)w->K, (int)w->Np);
}

cudaError_t launch_tensor(const tq2_weight* w, const float* x, float* out, int M, void* scratch,
                          cudaStream_t st, int bn_force, int splits_force) {
    const int N = (int)w->N, K = (int)w->K;
    const int tiles_n = (N + UM_BM - 1) / UM_BM;
    const int nk = K / UM_BK;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // The wide 384-token tile (a decoded stage feeds 1.5x the tokens, A in
    // tensor memory) only when its rounds of tiles cover fewer tokens than
    // those of 256-token tiles: per token the two run alike (163.9 against
    // 163.8 us at M=1536, N=27648, K=3072, both with A in tensor memory), and
    // the wide tile's coarser tiles can leave a last round half-empty (at
    // M=4096, N=14336: 313 against 285 us).
    int BN = umma_pick_bn(M);
    if (M >= UM_WIDE_BN) {
        const long long rounds_w = ((long long)tiles_n * ((M + UM_WIDE_BN - 1) / UM_WIDE_BN) + sms - 1) / sms;
        const long long rounds_n = ((long long)tiles_n * ((M + UM_MAX_BN - 1) / UM_MAX_BN) + sms - 1) / sms;
        if (rounds_w * UM_WIDE_BN < rounds_n * UM_MAX_BN) BN = UM_WIDE_BN;
    }
    if (bn_force > 0) BN = bn_force;
    const int tiles_m = (M + BN - 1) / BN;
    // K splits: 1 or 2 (two partials add into a zeroed output in either
    // order to the same sum); two only when they shorten the longest walk of
    // a CTA over its units of work by a quarter or more: the
    // atomic epilogue reads and writes the output twice (at M=4096 x
    // N=14336 a 6 % shorter walk cost 28 % more time)
    const int slots = sms, units1 = tiles_n * tiles_m;
    auto longest = [&](int sp) { return ((units1 * sp + slots - 1) / slots) * ((nk + sp - 1) / sp); };
    const int splits = splits_force > 0 ? splits_force : ((nk >= 4 && 4 * longest(2) <= 3 * longest(1)) ? 2 : 1);

    uint32_t* xh = reinterpret_cast<uint32_t*>(scratch);
    const int64_t groups = (int64_t)M * (K / 16);
    int64_t blocks = (groups + 255) / 256;
    if (blocks > 4 * (int64_t)sms * 8) blocks = 4 * (int64_t)sms * 8;
    if (blocks < 1) blocks = 1;
    cudaError_t e = launch_pdl(stage_x_f16_kernel, dim3((unsigned)blocks), dim3(256), 0, st, x, xh, (int64_t)M,
                               (int64_t)K, out, splits > 1 ? (int64_t)M * N : (int64_t)0);
    if (e != cudaSuccess) return e;

    EpiArgs ep{out, nullptr, nullptr, nullptr, nullptr, (int64_t)N, 1.0f};
    if (splits > 1) return launch_umma<DecTQ2, EPI_ATOMIC>(w->umma_maps, ep, xh, M, N, K, BN, splits, st);
    return launch_umma<DecTQ2, EPI_STORE>(w->umma_maps, ep, xh, M, N, K, BN, 1, st);
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
