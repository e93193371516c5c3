// api.cu -- the C ABI declared in include/tq2.h: argument checking, device
// memory of the weight handles, scratch from the stream-ordered allocator,
// kernel dispatch and status reporting.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "../../include/tq2.h"
#include "tq2_internal.h"
#include "tq2_quant.h"

namespace {

thread_local std::string g_last_error;

tq2_status fail(tq2_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

tq2_status cuda_fail(cudaError_t e, const char* what) {
    return fail(e == cudaErrorMemoryAllocation ? TQ2_ENOMEM : TQ2_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

inline cudaStream_t S(void* s) { return reinterpret_cast<cudaStream_t>(s); }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

}  // namespace

namespace tq2 {

int set_error(int st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

bool make_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, uint64_t inner, uint64_t outer,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dtype, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, const uint64_t (&dims)[3],
                        const uint64_t (&strides)[2], const uint32_t (&box)[3], CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
    const cuuint64_t st[2] = {strides[0], strides[1]};
    const cuuint32_t b[3] = {box[0], box[1], box[2]};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, dtype, 3, base, d, st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tq2

extern "C" {

const char* tq2_status_string(int status) {
    switch (status) {
        case TQ2_OK: return "ok";
        case TQ2_EINVAL: return "invalid argument";
        case TQ2_ESHAPE: return "shape not supported";
        case TQ2_ENOMEM: return "out of memory";
        case TQ2_ECUDA: return "CUDA error";
        case TQ2_ETIMEOUT: return "device-side wait timed out";
        case TQ2_EUNSUPPORTED: return "unsupported device or configuration";
        default: return "unknown status";
    }
}

const char* tq2_last_error(void) { return g_last_error.c_str(); }

const char* tq2_version(void) { return "tq2-gb300 sm_103a"; }

tq2_status tq2_device_status(void* stream) {
    cudaError_t e = cudaStreamSynchronize(S(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tq2_device_status: stream");
    const unsigned int err = tq2::read_clear_dev_error_skinny(S(stream)) | tq2::read_clear_dev_error_umma(S(stream)) |
                             tq2::read_clear_dev_error_blr(S(stream)) | tq2::read_clear_dev_error_gemv(S(stream));
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "tq2_device_status");
    if (err) return fail(TQ2_ETIMEOUT, "a bounded device-side wait ran out (record 0x%x)", err);
    return TQ2_OK;
}

tq2_status tq2_upload(const void* aos, int64_t N, int64_t K, tq2_handle* out, void* stream) {
    if (out) *out = nullptr;
    if (!aos || !out) return fail(TQ2_EINVAL, "tq2_upload: null pointer");
    if (N < 1 || K < 128 || K % 128 != 0) return fail(TQ2_ESHAPE, "tq2_upload: need N >= 1, K >= 128, K %% 128 == 0 (N=%lld K=%lld)", (long long)N, (long long)K);
    if (N > (int64_t)1 << 31 || K > (int64_t)1 << 30 || N * K >= (int64_t)1 << 40)
        return fail(TQ2_ESHAPE, "tq2_upload: weight too large");
    const int64_t nblocks = N * (K / 128);
    const size_t aos_bytes = (size_t)nblocks * 34;
    cudaStream_t st = S(stream);
    tq2_weight* w = new (std::nothrow) tq2_weight();
    if (!w) return fail(TQ2_ENOMEM, "tq2_upload: host allocation");
    w->N = N;
    w->K = K;
    w->Np = (N + 127) / 128 * 128;
    cudaGetDevice(&w->device);
    // Both planes carry a little zeroed padding: the GEMV's TMA box may run up
    // to 128 bytes past the last row's codes, its scale copy up to 14 bytes.
    cudaError_t e = cudaMalloc(&w->codes, (size_t)(N * K / 4) + 128);
    if (e == cudaSuccess) e = cudaMemset(w->codes + N * K / 4, 0, 128);
    if (e == cudaSuccess) e = cudaMalloc(&w->scales, (size_t)nblocks * 2 + 16);
    if (e == cudaSuccess) e = cudaMemset(w->scales + nblocks, 0, 16);
    if (e == cudaSuccess) e = cudaMalloc(&w->scales_t, (size_t)(K / 128) * w->Np * 2);
    if (e == cudaSuccess) e = cudaMalloc(&w->codes_t, (size_t)(K / 4) * w->Np);
    auto release = [w]() {
        cudaFree(w->codes);
        cudaFree(w->scales);
        cudaFree(w->scales_t);
        cudaFree(w->codes_t);
        delete w;
    };
    if (e != cudaSuccess) {
        release();
        return cuda_fail(e, "tq2_upload: cudaMalloc");
    }
    uint8_t* tmp = nullptr;
    e = cudaMallocAsync(reinterpret_cast<void**>(&tmp), aos_bytes, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(tmp, aos, aos_bytes, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = tq2::launch_repack(tmp, w->codes, w->scales, nblocks, st);
    if (e == cudaSuccess) e = tq2::launch_scales_t(w->scales, w->scales_t, N, K / 128, w->Np, st);
    if (e == cudaSuccess) e = tq2::launch_codes_t(w->codes, w->codes_t, N, K, w->Np, st);
    if (tmp) cudaFreeAsync(tmp, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        release();
        return cuda_fail(e, "tq2_upload");
    }
    if (!tq2::make_gemv_maps(w) || !tq2::make_umma_maps(w)) {
        release();
        return fail(TQ2_EUNSUPPORTED, "tq2_upload: cuTensorMapEncodeTiled refused a code-plane map");
    }
    *out = w;
    return TQ2_OK;
}

tq2_status tq2_free(tq2_handle h) {
    if (!h) return TQ2_OK;
    cudaError_t e1 = cudaFree(h->codes);
    cudaError_t e2 = cudaFree(h->scales);
    cudaError_t e3 = cudaFree(h->scales_t);
    cudaError_t e4 = cudaFree(h->codes_t);
    delete h;
    if (e4 != cudaSuccess) return cuda_fail(e4, "tq2_free");
    if (e3 != cudaSuccess) return cuda_fail(e3, "tq2_free");
    if (e1 != cudaSuccess) return cuda_fail(e1, "tq2_free");
    if (e2 != cudaSuccess) return cuda_fail(e2, "tq2_free");
    return TQ2_OK;
}

tq2_status tq2_shape(tq2_handle h, int64_t* N, int64_t* K) {
    if (!h || !N || !K) return fail(TQ2_EINVAL, "tq2_shape: null pointer");
    *N = h->N;
    *K = h->K;
    return TQ2_OK;
}

tq2_status tq2_gemm_path(tq2_handle h, const float* x, float* out, int64_t M, int64_t N, int64_t K, int path,
                         void* stream) {
    if (!h) return fail(TQ2_EINVAL, "tq2_gemm: null handle");
    if (M == 0) return TQ2_OK;
    if (!x || !out) return fail(TQ2_EINVAL, "tq2_gemm: null pointer");
    if (M < 0 || M > (int64_t)1 << 24) return fail(TQ2_ESHAPE, "tq2_gemm: bad M=%lld", (long long)M);
    if (N != h->N || K != h->K)
        return fail(TQ2_ESHAPE, "tq2_gemm: (N,K)=(%lld,%lld) but the handle holds (%lld,%lld)", (long long)N,
                    (long long)K, (long long)h->N, (long long)h->K);
    if ((reinterpret_cast<uintptr_t>(x) & 15) != 0) return fail(TQ2_EINVAL, "tq2_gemm: x must be 16-byte aligned");
    if (path == TQ2_PATH_AUTO) path = M <= 16 ? TQ2_PATH_SKINNY : TQ2_PATH_TENSOR;
    cudaStream_t st = S(stream);
    if (path == TQ2_PATH_SKINNY) {
        if (M > 16) return fail(TQ2_ESHAPE, "tq2_gemm: skinny kernel needs M <= 16");
        if (tq2::gemv_supports((int)M, K)) {   // fused single-kernel GEMV, no scratch
            cudaError_t e = tq2::launch_gemv(&h, &x, &out, 1, (int)M, st);
            if (e != cudaSuccess) return cuda_fail(e, "tq2_gemm: gemv launch");
            return TQ2_OK;
        }
        void* scratch = nullptr;
        cudaError_t e = cudaMallocAsync(&scratch, tq2::skinny_scratch_bytes(M, K), st);
        if (e != cudaSuccess) return cuda_fail(e, "tq2_gemm: scratch");
        e = tq2::launch_skinny(h->codes, h->scales, x, out, (int)M, (int)N, (int)K, scratch, st);
        cudaError_t e2 = cudaFreeAsync(scratch, st);
        if (e != cudaSuccess) return cuda_fail(e, "tq2_gemm: skinny launch");
        if (e2 != cudaSuccess) return cuda_fail(e2, "tq2_gemm: scratch free");
        return TQ2_OK;
    }
    if (path == TQ2_PATH_TENSOR) {
        if (M * K >= (int64_t)1 << 31) return fail(TQ2_ESHAPE, "tq2_gemm: M*K too large for the tensor path");
        void* scratch = nullptr;
        cudaError_t e = cudaMallocAsync(&scratch, tq2::tensor_scratch_bytes(M, K), st);
        if (e != cudaSuccess) return cuda_fail(e, "tq2_gemm: scratch");
        e = tq2::launch_tensor(h, x, out, (int)M, scratch, st);
        cudaError_t e2 = cudaFreeAsync(scratch, st);
        if (e != cudaSuccess) return cuda_fail(e, "tq2_gemm: tensor launch");
        if (e2 != cudaSuccess) return cuda_fail(e2, "tq2_gemm: scratch free");
        return TQ2_OK;
    }
    return fail(TQ2_EINVAL, "tq2_gemm: unknown path %d", path);
}

tq2_status tq2_gemm_tensor_tuned(tq2_handle h, const float* x, float* out, int64_t M, int64_t N, int64_t K,
                                 int bn, int splits, void* stream) {
    if (!h) return fail(TQ2_EINVAL, "tq2_gemm_tensor_tuned: null handle");
    if (M == 0) return TQ2_OK;
    if (!x || !out) return fail(TQ2_EINVAL, "tq2_gemm_tensor_tuned: null pointer");
    if (M < 0 || M > (int64_t)1 << 24 || M * K >= (int64_t)1 << 31)
        return fail(TQ2_ESHAPE, "tq2_gemm_tensor_tuned: bad M=%lld", (long long)M);
    if (N != h->N || K != h->K)
        return fail(TQ2_ESHAPE, "tq2_gemm_tensor_tuned: (N,K)=(%lld,%lld) but the handle holds (%lld,%lld)",
                    (long long)N, (long long)K, (long long)h->N, (long long)h->K);
    if ((reinterpret_cast<uintptr_t>(x) & 15) != 0)
        return fail(TQ2_EINVAL, "tq2_gemm_tensor_tuned: x must be 16-byte aligned");
    // token tile: a multiple of 16 up to 256 (one that is not a multiple of
    // 32 must cover all M tokens), or 384 with N > 128; K splits: 1..16
    // and at most K/64
    const bool wide = bn == 384 && N > 128;
    if (bn != 0 && !wide && (bn < 16 || bn > 256 || bn % 16 != 0 || (bn % 32 != 0 && M > bn)))
        return fail(TQ2_EINVAL, "tq2_gemm_tensor_tuned: bad token tile %d", bn);
    if (splits != 0 && (splits < 1 || splits > 16 || splits > K / 64))
        return fail(TQ2_EINVAL, "tq2_gemm_tensor_tuned: bad split count %d", splits);
    cudaStream_t st = S(stream);
    void* scratch = nullptr;
    cudaError_t e = cudaMallocAsync(&scratch, tq2::tensor_scratch_bytes(M, K), st);
    if (e != cudaSuccess) return cuda_fail(e, "tq2_gemm_tensor_tuned: scratch");
    e = tq2::launch_tensor(h, x, out, (int)M, scratch, st, bn, splits);
    cudaError_t e2 = cudaFreeAsync(scratch, st);
    if (e != cudaSuccess) return cuda_fail(e, "tq2_gemm_tensor_tuned: launch");
    if (e2 != cudaSuccess) return cuda_fail(e2, "tq2_gemm_tensor_tuned: scratch free");
    return TQ2_OK;
}

tq2_status tq2_gemm(tq2_handle h, const float* x, float* out, int64_t M, int64_t N, int64_t K, void* stream) {
    return tq2_gemm_path(h, x, out, M, N, K, TQ2_PATH_AUTO, stream);
}

tq2_status tq2_gemm_grouped(const tq2_handle* hs, const float* const* xs, float* const* outs, int G, int64_t M,
                            int64_t K, void* stream) {
    if (!hs || !xs || !outs) return fail(TQ2_EINVAL, "tq2_gemm_grouped: null array");
    if (G < 1 || G > tq2::GEMV_MAX_JOBS) return fail(TQ2_ESHAPE, "tq2_gemm_grouped: need 1 <= G <= %d", tq2::GEMV_MAX_JOBS);
    if (!tq2::gemv_supports((int)M, K))
        return fail(TQ2_ESHAPE,
                    "tq2_gemm_grouped: need 1 <= M <= %d and MT*K <= %lld, MT = M rounded up to 1, 2, 4 or 8 "
                    "(M=%lld K=%lld)",
                    tq2::GEMV_MAX_M, (long long)tq2::GEMV_MAX_MK, (long long)M, (long long)K);
    int64_t rows = 0;
    for (int g = 0; g < G; ++g) {
        const tq2_handle h = hs[g];
        if (!h || !xs[g] || !outs[g]) return fail(TQ2_EINVAL, "tq2_gemm_grouped: null entry %d", g);
        if (h->K != K) return fail(TQ2_ESHAPE, "tq2_gemm_grouped: entry %d has K=%lld, not %lld", g, (long long)h->K, (long long)K);
        if ((reinterpret_cast<uintptr_t>(xs[g]) & 15) != 0) return fail(TQ2_EINVAL, "tq2_gemm_grouped: x %d not 16-byte aligned", g);
        rows += h->N;
    }
    if (rows >= ((int64_t)1 << 31)) return fail(TQ2_ESHAPE, "tq2_gemm_grouped: too many rows");
    cudaError_t e = tq2::launch_gemv(hs, xs, outs, G, (int)M, S(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tq2_gemm_grouped");
    return TQ2_OK;
}

tq2_status tq2_unpack(tq2_handle h, void* aos_out, void* stream) {
    if (!h || !aos_out) return fail(TQ2_EINVAL, "tq2_unpack: null pointer");
    const int64_t nblocks = h->N * (h->K / 128);
    const size_t bytes = (size_t)nblocks * 34;
    cudaStream_t st = S(stream);
    uint8_t* tmp = nullptr;
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&tmp), bytes, st);
    if (e == cudaSuccess) e = tq2::launch_unpack(h->codes, h->scales, tmp, nblocks, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(aos_out, tmp, bytes, cudaMemcpyDeviceToHost, st);
    if (tmp) cudaFreeAsync(tmp, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "tq2_unpack");
    return TQ2_OK;
}

tq2_status tq2_quantize(const float* w, int64_t N, int64_t K, void* aos_out, void* stream) {
    if (!w || !aos_out) return fail(TQ2_EINVAL, "tq2_quantize: null pointer");
    if (N < 1 || K < 128 || K % 128 != 0)
        return fail(TQ2_ESHAPE, "tq2_quantize: need N >= 1, K >= 128, K %% 128 == 0 (N=%lld K=%lld)", (long long)N,
                    (long long)K);
    if (N > ((int64_t)1 << 40) / K) return fail(TQ2_ESHAPE, "tq2_quantize: weight too large");
    cudaError_t e = tq2::launch_quantize(w, static_cast<uint8_t*>(aos_out), N, K, S(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tq2_quantize");
    return TQ2_OK;
}

tq2_status tq2_dequant_f16(tq2_handle h, uint16_t* w, void* stream) {
    if (!h || !w) return fail(TQ2_EINVAL, "tq2_dequant_f16: null pointer");
    cudaError_t e = tq2::launch_dequant_f16(h->codes, h->scales, w, h->N, h->K, S(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tq2_dequant_f16");
    return TQ2_OK;
}

}  // extern "C"
