// tq2_internal.h -- declarations shared by the library's translation units
// (host side only).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tq2 {
// Tensor maps of a plane for the tcgen05 core (umma_core.cuh).
struct PlaneMaps {
    CUtensorMap m0, m1;
};
}  // namespace tq2

struct tq2_weight {
    int64_t N = 0, K = 0;
    int64_t Np = 0;                // N rounded up to a multiple of 128
    uint8_t* codes = nullptr;      // [N][K/4], then 128 bytes of padding
    uint16_t* scales = nullptr;    // [N][K/128] f16 bits, then 16 bytes of padding
    uint16_t* scales_t = nullptr;  // [K/128][Np] the same bits block-major (rows >= N zero), for the tensor path
    uint8_t* codes_t = nullptr;    // [Np/128][K/64][128 rows][16 B] the same codes stage-tiled (rows >= N zero),
                                   // for the tensor path: one K-stage of a 128-row tile is 2 KB contiguous
    int device = 0;
    // 3D views of the code plane for the GEMV's TMA loads, built at upload:
    // (128-byte piece, row, piece index), strides (1, K/4, 128) bytes; boxes
    // of 16 rows x 8 pieces (k-split units) and 128 rows x 1 piece (row units).
    CUtensorMap gemv_map_k, gemv_map_r;
    // the tensor path's views: 2 KB code stages of the stage-tiled copy and
    // block-major scale rows of 128 (umma_core.cuh, plane_maps_tq2)
    tq2::PlaneMaps umma_maps;
};

namespace tq2 {

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel on the stream drains; it must call griddepcontrol.wait
// before touching anything that earlier work writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// tq2_skinny.cu
cudaError_t launch_repack(const uint8_t* aos_dev, uint8_t* codes, uint16_t* scales, int64_t nblocks,
                          cudaStream_t st);
cudaError_t launch_unpack(const uint8_t* codes, const uint16_t* scales, uint8_t* aos_dev, int64_t nblocks,
                          cudaStream_t st);
cudaError_t launch_scales_t(const uint16_t* scales, uint16_t* scales_t, int64_t N, int64_t nb, int64_t Np,
                            cudaStream_t st);
cudaError_t launch_codes_t(const uint8_t* codes, uint8_t* codes_t, int64_t N, int64_t K, int64_t Np, cudaStream_t st);
cudaError_t launch_dequant_f16(const uint8_t* codes, const uint16_t* scales, uint16_t* w, int64_t N,
                               int64_t K, cudaStream_t st);
size_t skinny_scratch_bytes(int64_t M, int64_t K);
cudaError_t launch_skinny(const uint8_t* codes, const uint16_t* scales, const float* x, float* out, int M,
                          int N, int K, void* scratch, cudaStream_t st);
unsigned int read_clear_dev_error_skinny(cudaStream_t st);

// tq2_gemv.cu: fused GEMV for M <= GEMV_MAX_M and MT*K <= GEMV_MAX_MK, MT = M
// rounded up to 1, 2, 4 or 8 (no
// scratch; x lives in shared memory); one launch runs G <= GEMV_MAX_JOBS
// independent GEMVs of the same K and M.
constexpr int GEMV_MAX_M = 8;
constexpr int64_t GEMV_MAX_MK = 32768;
constexpr int GEMV_MAX_JOBS = 64;
bool gemv_supports(int M, int64_t K);
bool make_gemv_maps(tq2_weight* w);
cudaError_t launch_gemv(const tq2_weight* const* ws, const float* const* xs, float* const* outs, int G, int M,
                        cudaStream_t st);
unsigned int read_clear_dev_error_gemv(cudaStream_t st);

// tq2_umma.cu
bool make_umma_maps(tq2_weight* w);
size_t tensor_scratch_bytes(int64_t M, int64_t K);
cudaError_t launch_tensor(const tq2_weight* w, const float* x, float* out, int M, void* scratch,
                          cudaStream_t st, int bn_force = 0,
                          int splits_force = 0);
unsigned int read_clear_dev_error_umma(cudaStream_t st);

// blr_rank.cu: res = oscale * f16(act . vec * scale) P over the sign plane of
// `bits` ([K][r/32], the plane's row index as the GEMM's K), f16 staging of
// res * col * scale2 for the next GEMM, optional column sums of res * other.
cudaError_t launch_blr_rank(const float* act, const float* vec, float scale, const uint32_t* bits, int T, int K,
                            int r, float oscale, float* res, const float* col, float scale2, uint16_t* st16,
                            const float* other, float* colpart, cudaStream_t st);

// blr.cu
cudaError_t launch_expand_bits(const uint32_t* bits, int64_t rows, int64_t r, uint16_t* plane, int transpose,
                               cudaStream_t st);
unsigned int read_clear_dev_error_blr(cudaStream_t st);

// api.cu: record the calling thread's last error message; returns `st`.
int set_error(int st, const char* fmt, ...);

// tensor maps (api.cu): 2D tiled map, inner dimension first.
bool make_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, uint64_t inner,
                        uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                        CUtensorMapSwizzle swizzle);
// 3D tiled map: dims[0] innermost (unit stride), strides of dims 1 and 2 in bytes.
bool make_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, const uint64_t (&dims)[3],
                        const uint64_t (&strides)[2], const uint32_t (&box)[3], CUtensorMapSwizzle swizzle);

}  // namespace tq2
