// blr.cu -- binary low-rank layer ("cortiq-engine 0.8.43, src/gpu_wgpu/
// train_mm.rs"): sign-bitmap expansion and the layer's forward / backward.
//
// Bitmap convention (kernels expand / expand_n / expand_t on that page):
// bits [rows][r/32] u32, bit j of word w is rank 32w + j, a set bit is +1.
#include "../../include/tq2.h"
#include "ptx.cuh"
#include "tq2_internal.h"

namespace tq2 {

// One thread per output element; f16 +-1 = 0x3C00 with the sign bit set
// for a clear bit.
__global__ void expand_bits_kernel(const uint32_t* __restrict__ bits, int64_t rows, int64_t r,
                                   uint16_t* __restrict__ plane, int transpose) {
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= rows * r) return;
    int64_t row, k;
    if (transpose) {        // plane[k][row], consecutive threads along rows
        k = i / rows;
        row = i % rows;
    } else {                // plane[row][k]
        row = i / r;
        k = i % r;
    }
    const uint32_t b = (bits[row * (r / 32) + k / 32] >> (k % 32)) & 1u;
    plane[i] = (uint16_t)(0x3C00u | ((b ^ 1u) << 15));
}

cudaError_t launch_expand_bits(const uint32_t* bits, int64_t rows, int64_t r, uint16_t* plane, int transpose,
                               cudaStream_t st) {
    const int64_t n = rows * r;
    expand_bits_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(bits, rows, r, plane, transpose);
    return cudaGetLastError();
}

unsigned int read_clear_dev_error_blr(cudaStream_t st) {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_dev_error, sizeof(v), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return 0;
    cudaMemcpyToSymbolAsync(g_dev_error, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
    cudaStreamSynchronize(st);
    return v;
}

}  // namespace tq2

namespace {
tq2_status blr_fail(tq2_status st, const char* msg) { return (tq2_status)tq2::set_error(st, "%s", msg); }
}  // namespace

extern "C" {

tq2_status blr_expand_bits(const uint32_t* bits, int64_t rows, int64_t r, uint16_t* plane_f16, int transpose,
                           void* stream) {
    if (!bits || !plane_f16) return blr_fail(TQ2_EINVAL, "blr_expand_bits: null pointer");
    if (rows < 1 || r < 32 || r % 32 != 0) return blr_fail(TQ2_ESHAPE, "blr_expand_bits: need rows >= 1, r % 32 == 0");
    cudaError_t e = tq2::launch_expand_bits(bits, rows, r, plane_f16, transpose, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TQ2_OK : TQ2_ECUDA;
}

tq2_status blr_forward(const uint32_t*, const uint32_t*, const float*, const float*, const float*, const float*,
                       float*, float*, float*, int64_t, int64_t, int64_t, int64_t, void*) {
    return blr_fail(TQ2_EUNSUPPORTED, "blr_forward: not built yet");
}

tq2_status blr_backward(const uint32_t*, const uint32_t*, const float*, const float*, const float*, const float*,
                        const float*, const float*, const float*, float*, float*, float*, float*, int64_t, int64_t,
                        int64_t, int64_t, float, void*) {
    return blr_fail(TQ2_EUNSUPPORTED, "blr_backward: not built yet");
}

}  // extern "C"
