// tq2_quant.cu -- the ternary producer: f32 weights -> BlockTQ2_0_g128 blocks.
//
// Per 128-element block of a weight row, the 2-bit fake-quantize of
// "rlx-mlx 0.2.13, src/lower/helpers.rs" (fq_q_max: 2 bits -> q_max = 1;
// fq_scale_perbatch: max|w| / q_max floored at 1e-12; fq_quantize_dequantize:
// round, clamp to [-q_max, q_max]), all in f32:
//   s    = max(max_k |w_k|, 1e-12)
//   q_k  = clamp(round_half_even(w_k / s), -1, 1)      (IEEE f32 division)
//   code = q_k + 1,   d = f16(s) (nearest, ties to even)
// stored as the pages' AoS block { qs[32], d } (34 bytes; code of element
// 4j+i in bits 2i..2i+1 of qs[j]; "oxibonsai-kernels 0.2.1,
// src/gpu_backend/metal_graph/tests_gemm_tq2.rs").
//
// One warp per block: lane j loads elements 4j..4j+3 (one 16-byte load, the
// warp's 512 bytes coalesced), the block maximum is a shuffle reduction
// (exact), lane j writes qs[j] and lane 0 writes d.  Each warp takes two
// blocks per pass with both loads issued first, so enough bytes are in
// flight to stream HBM: 512 bytes read and 34 written per block.
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "tq2_internal.h"
#include "tq2_quant.h"

namespace tq2 {

namespace {

__device__ __forceinline__ void quant_block(const float4 v, uint8_t* blk, int lane) {
    float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float s = fmaxf(m, 1e-12f);                  // max|w| / q_max with q_max = 1
    // round(w / s) in {-1, 0, +1} decided without the division.  With
    // |w| <= s, the correctly rounded quotient exceeds 0.5 exactly when
    // w / s > 0.5 + 2^-25 (the midpoint between 0.5 and the next float above
    // it ties to the even 0.5), i.e. when w - s/2 > s * 2^-25.  Both s/2 and
    // s * 2^-25 are exact (s >= 1e-12 is normal), and w - s/2 is exact for
    // s/4 <= w <= s (Sterbenz); for smaller w it is negative anyway.  So the
    // code is the one round-half-even(w / s) gives, for every finite w.
    const float h = 0.5f * s, e = s * 0x1p-25f;
    auto code = [&](float w) -> uint32_t { return w - h > e ? 2u : (-w - h > e ? 0u : 1u); };
    blk[lane] = (uint8_t)(code(v.x) | (code(v.y) << 2) | (code(v.z) << 4) | (code(v.w) << 6));
    // d, little endian: one 16-bit store (a block starts at an even offset)
    if (lane == 0) *reinterpret_cast<uint16_t*>(blk + 32) = __half_as_ushort(__float2half_rn(s));
}

__global__ void __launch_bounds__(256) quantize_kernel(const float* __restrict__ w, uint8_t* __restrict__ aos,
                                                       int64_t nblocks) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    // blocks warp0, warp0 + nwarps, ... taken two at a time
    for (int64_t b = warp0; b < nblocks; b += 2 * nwarps) {
        const int64_t b2 = b + nwarps;
        const float4 v0 = __ldg(reinterpret_cast<const float4*>(w + b * 128) + lane);
        const float4 v1 = b2 < nblocks ? __ldg(reinterpret_cast<const float4*>(w + b2 * 128) + lane)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
        quant_block(v0, aos + b * 34, lane);
        if (b2 < nblocks) quant_block(v1, aos + b2 * 34, lane);   // warp-uniform
    }
}

}  // namespace

cudaError_t launch_quantize(const float* w, uint8_t* aos, int64_t N, int64_t K, cudaStream_t st) {
    const int64_t nblocks = N * (K / 128);
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // 8 warps per CTA, 8 CTAs per SM; each warp takes blocks in pairs
    int64_t grid = (nblocks + 15) / 16;
    if (grid > (int64_t)sms * 8) grid = (int64_t)sms * 8;
    if (grid < 1) grid = 1;
    quantize_kernel<<<(unsigned)grid, 256, 0, st>>>(w, aos, nblocks);
    return cudaGetLastError();
}

}  // namespace tq2
