// blr.cu -- binary low-rank layer ("cortiq-engine 0.8.43, src/gpu_wgpu/
// train_mm.rs"): sign-bitmap expansion and one path's forward / backward.
//
//   W = diag(h) S_U diag(l) S_V^T diag(g)         (module doc)
//   forward   a = (x.g) S_V      c = (a.l) S_U^T      y = h.c
//   backward  dh += sum_t dy.c   b = (dy.h) S_U       dl += sum_t a.b
//             dx' = (b.l) S_V^T  dg += sum_t x.dx'    dx = g.dx'
//
// Bitmap convention (kernels expand / expand_n / expand_t on that page):
// bits [rows][r/32] u32, bit j of word w is rank 32w + j, a set bit is +1.
//
// GPU mapping.  The two products that contract over d_in or d_out and land
// in rank space (a, b) run in blr_rank.cu: one pass over the f32 activation,
// rounded to f16 on chip, times the sign plane read in its own row order,
// reduced over a cluster in a fixed order.  The two that expand rank space
// back to d_out or d_in (c, dx') are tcgen05 GEMMs on the core
// (umma_core.cuh) with the sign plane decoded on chip (DecSign, the bits as
// given) and the f16 rank-space operand staged by the rank kernel:
//   a  : f16(x.g)        x S_V        K = d_in    (blr_rank.cu; also a_save, f16(a.l))
//   c  : f16(a.l)        x S_U^T      K = r       (core; y = h.c in the epilogue)
//   b  : f16(dy.h.gs)    x S_U  / gs  K = d_out   (blr_rank.cu; f16(b.l.gs), dl partials)
//   dx': f16(b.l.gs)     x S_V^T / gs K = r       (core; dx = g.dx', dg partials)
// The column sums dh, dl, dg are two-pass reductions in a fixed order
// (partials per token tile or 32-token chunk, then an ordered sum), so every
// result is deterministic.  gs (a power of two) keeps staged gradients away
// from the f16 subnormals; the GEMMs divide it back out.
#include <cmath>

#include "../../include/tq2.h"
#include "tq2_internal.h"
#include "umma_core.cuh"

namespace tq2 {

// ------------------------------------------------------------ expansion ----
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

// ------------------------------------------------------------- staging ----
// dst[t][k] f16 = f16((src[t][k] * col[k]) * scale) in the 32-group pair
// order of DecSign (position 2p = element p, 2p+1 = element p+16).  One
// thread per quarter q of a 32-element group: it reads elements 4q..4q+3 and
// 16+4q..16+4q+3 (two float4) and writes pair words 4q..4q+3 (one uint4), so
// a warp touches 8 whole 128-byte groups per pair of loads.
__global__ void stage32_kernel(const float* __restrict__ src, const float* __restrict__ col, float scale,
                               uint32_t* __restrict__ dst, int64_t T, int64_t Kd) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t quarters = T * (Kd / 32) * 4;
    for (int64_t qi = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; qi < quarters;
         qi += (int64_t)gridDim.x * blockDim.x) {
        const int64_t gi = qi >> 2;
        const int q = (int)(qi & 3);
        const int64_t t = gi / (Kd / 32), k0 = (gi % (Kd / 32)) * 32;
        const float* sp = src + t * Kd + k0;
        float4 lo = *reinterpret_cast<const float4*>(sp + 4 * q);
        float4 hi = *reinterpret_cast<const float4*>(sp + 16 + 4 * q);
        if (col) {
            const float4 cl = *reinterpret_cast<const float4*>(col + k0 + 4 * q);
            const float4 ch = *reinterpret_cast<const float4*>(col + k0 + 16 + 4 * q);
            lo.x *= cl.x; lo.y *= cl.y; lo.z *= cl.z; lo.w *= cl.w;
            hi.x *= ch.x; hi.y *= ch.y; hi.z *= ch.z; hi.w *= ch.w;
        }
        uint32_t o[4];
        const float l4[4] = {lo.x, lo.y, lo.z, lo.w}, h4[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 h = __floats2half2_rn(l4[i] * scale, h4[i] * scale);
            o[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        reinterpret_cast<uint4*>(dst + (t * Kd + k0) / 2)[q] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// Tokens per partial column sum (a chunk) of the colsum kernels.
constexpr int FIN_TC = 32;

// dst[c][t] = f16(src[t][c] * col[c] * scale) for t < T and 0 for T <= t < Tp:
// an operand of a GEMM over the token axis, transposed so that the tokens
// are its K (natural order, as both TMA-loaded operands of the core expect).
// 64 x 64 tiles through shared memory, 256 threads: 16-byte loads along c
// (16 threads a token row), 4-byte stores of two tokens along t (32 threads,
// 128 bytes, a c row).  C is a multiple of 64 (d_in, d_out, r).
__global__ void __launch_bounds__(256) stage_t16_kernel(const float* __restrict__ src, int T, int C,
                                                        const float* __restrict__ col, float scale,
                                                        uint16_t* __restrict__ dst, int Tp) {
    __shared__ float tile[64][65];
    pdl_wait();
    pdl_launch_dependents();
    const int c0 = blockIdx.x * 64, t0 = blockIdx.y * 64, tid = threadIdx.x;
    {
        const int cq = (tid & 15) * 4, tr = tid >> 4;                  // 4 columns, token row 0..15
        const float4 cv = *reinterpret_cast<const float4*>(col + c0 + cq);
#pragma unroll
        for (int pass = 0; pass < 4; ++pass) {
            const int i = tr + 16 * pass, t = t0 + i;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < T) v = *reinterpret_cast<const float4*>(src + (int64_t)t * C + c0 + cq);
            tile[i][cq] = v.x * cv.x;
            tile[i][cq + 1] = v.y * cv.y;
            tile[i][cq + 2] = v.z * cv.z;
            tile[i][cq + 3] = v.w * cv.w;
        }
    }
    __syncthreads();
    {
        const int tp = (tid & 31) * 2, cr = tid >> 5;                  // two tokens, c row 0..7
#pragma unroll
        for (int pass = 0; pass < 8; ++pass) {
            const int j = cr + 8 * pass, c = c0 + j, t = t0 + tp;
            if (t < Tp) {
                const __half2 h2 = __floats2half2_rn(tile[tp][j] * scale, tile[tp + 1][j] * scale);
                *reinterpret_cast<__half2*>(dst + (int64_t)c * Tp + t) = h2;
            }
        }
    }
}

// colpart[chunk][n] = sum over the chunk's tokens of A[t][n] * B[t][n]
// (block (32, 8): x = column within a 32-column group, y = token lane; fixed
// order).
__global__ void colsum_prod_kernel(const float* __restrict__ A, const float* __restrict__ B, int T, int n,
                                   float* __restrict__ colpart) {
    __shared__ float red[8][33];
    pdl_wait();
    pdl_launch_dependents();
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int j = blockIdx.x * 32 + tx;
    const int t0 = blockIdx.y * FIN_TC;
    float acc = 0.f;
    if (j < n)
        for (int t = t0 + ty; t < t0 + FIN_TC && t < T; t += 8)
            acc = fmaf(A[(int64_t)t * n + j], B[(int64_t)t * n + j], acc);
    red[ty][tx] = acc;
    __syncthreads();
    if (ty == 0 && j < n) {
        float s2 = 0.f;
        for (int i = 0; i < 8; ++i) s2 += red[i][tx];
        colpart[(int64_t)blockIdx.y * n + j] = s2;
    }
}

// The backward's three column sums in one launch: job blockIdx.y of
// {dh, dl, dg}, out[n] += sum_c colpart[c][n], c in order (the same order and
// arithmetic for each of the three).
struct ColsumJobs {
    const float* colpart[3];
    int chunks[3], n[3];
    float* out[3];
};
__global__ void colsum_finish3_kernel(const ColsumJobs jobs) {
    pdl_wait();
    pdl_launch_dependents();
    const int q = blockIdx.y;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= jobs.n[q]) return;
    const float* cp = jobs.colpart[q];
    const int n = jobs.n[q], chunks = jobs.chunks[q];
    float s = 0.f;
    // in order, 16 partials loaded ahead of their additions (one memory
    // round trip per 16 instead of a dependent chain of loads)
    int c = 0;
    for (; c + 16 <= chunks; c += 16) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = cp[(int64_t)(c + i) * n + j];
#pragma unroll
        for (int i = 0; i < 16; ++i) s += v[i];
    }
    for (; c < chunks; ++c) s += cp[(int64_t)c * n + j];
    jobs.out[q][j] += s;
}

unsigned int read_clear_dev_error_blr(cudaStream_t st) {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_dev_error, sizeof(v), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return 0;
    cudaMemcpyToSymbolAsync(g_dev_error, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
    cudaStreamSynchronize(st);
    return v;
}

// ---------------------------------------------------------- host pieces ----
namespace {

struct Scratch {
    char* base = nullptr;
    size_t off = 0;
    template <class T>
    T* take(size_t n) {
        T* p = reinterpret_cast<T*>(base + off);
        off += (n * sizeof(T) + 255) & ~size_t(255);
        return p;
    }
};

int sm_count() {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

// Token tile of the layer's GEMMs: 256 tokens when there are enough (fewer
// tiles, so fewer per-tile fills and drains; measured faster at T = 2048
// than 128-token tiles with the sign plane in tensor memory), else all tokens.
int blr_bn(int T) { return umma_pick_bn(T); }

cudaError_t stage32(const float* src, const float* col, float scale, void* dst, int T, int Kd, cudaStream_t st) {
    const int64_t quarters = (int64_t)T * (Kd / 32) * 4;
    int64_t blocks = (quarters + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (blocks > cap) blocks = cap;
    return launch_pdl(stage32_kernel, dim3((unsigned)blocks), dim3(256), 0, st, src, col, scale,
                      reinterpret_cast<uint32_t*>(dst), (int64_t)T, (int64_t)Kd);
}

}  // namespace
}  // namespace tq2

// ---------------------------------------------------------------- C ABI ----
namespace {
using namespace tq2;

tq2_status blr_fail(tq2_status st, const char* msg) { return (tq2_status)set_error(st, "%s", msg); }

tq2_status check_shapes(const char* who, int64_t T, int64_t d_in, int64_t d_out, int64_t r) {
    if (T < 1 || d_in < 64 || d_out < 64 || r < 128 || d_in % 64 || d_out % 64 || r % 128)
        return (tq2_status)set_error(TQ2_ESHAPE,
                                     "%s: need T >= 1, d_in and d_out multiples of 64, r a multiple of 128 "
                                     "(T=%lld d_in=%lld d_out=%lld r=%lld)",
                                     who, (long long)T, (long long)d_in, (long long)d_out, (long long)r);
    const int64_t mx = d_in > d_out ? d_in : d_out;
    if (T * mx >= ((int64_t)1 << 31) || T * r * 8 >= ((int64_t)1 << 31) || mx > (1 << 20))
        return (tq2_status)set_error(TQ2_ESHAPE, "%s: problem too large", who);
    return TQ2_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

tq2_status cuda_status(cudaError_t e, const char* who) {
    if (e == cudaSuccess) return TQ2_OK;
    return (tq2_status)set_error(e == cudaErrorMemoryAllocation ? TQ2_ENOMEM : TQ2_ECUDA, "%s: %s", who,
                                 cudaGetErrorString(e));
}

}  // namespace

extern "C" {

tq2_status blr_expand_bits(const uint32_t* bits, int64_t rows, int64_t r, uint16_t* plane_f16, int transpose,
                           void* stream) {
    if (!bits || !plane_f16) return blr_fail(TQ2_EINVAL, "blr_expand_bits: null pointer");
    if (rows < 1 || r < 32 || r % 32 != 0) return blr_fail(TQ2_ESHAPE, "blr_expand_bits: need rows >= 1, r % 32 == 0");
    return cuda_status(launch_expand_bits(bits, rows, r, plane_f16, transpose, reinterpret_cast<cudaStream_t>(stream)),
                       "blr_expand_bits");
}

}  // extern "C"

namespace {

// One path forward; accumulate: y = fl(y + fl(h.c)) instead of y = fl(h.c).
// Arguments already checked.
tq2_status forward_one(const char* who, const uint32_t* bits_u, const uint32_t* bits_v, const float* h, const float* l,
                       const float* g, const float* x, float* y, float* a_save, float* c_save, int64_t T, int64_t d_in,
                       int64_t d_out, int64_t r, int accumulate, cudaStream_t st) {
    const int iT = (int)T, din = (int)d_in, dout = (int)d_out, ir = (int)r;
    void* al16 = nullptr;
    cudaError_t e = cudaMallocAsync(&al16, (size_t)T * r * 2, st);
    if (e != cudaSuccess) return cuda_status(e, who);
    // a = (x.g) S_V (one pass over x), a_save, and f16(a.l) for the next GEMM
    e = launch_blr_rank(x, g, 1.0f, bits_v, iT, din, ir, 1.0f, a_save, l, 1.0f, reinterpret_cast<uint16_t*>(al16),
                        nullptr, nullptr, st);
    if (e == cudaSuccess) {
        PlaneMaps pm;
        EpiArgs ep{y, c_save, h, nullptr, nullptr, (int64_t)d_out, 1.0f, accumulate};
        e = plane_maps_sign(pm, bits_u, dout, ir) ? launch_umma<DecSign, EPI_SCALE>(pm, ep, al16, iT, dout, ir,
                                                                                    blr_bn(iT), 1, st)
                                                  : cudaErrorInvalidValue;
    }
    cudaError_t e2 = cudaFreeAsync(al16, st);
    if (e != cudaSuccess) return cuda_status(e, who);
    return cuda_status(e2, who);
}

// One path backward; accumulate: dx = fl(dx + fl(g.dx')) instead of fl(g.dx').
// Arguments already checked.
tq2_status backward_one(const char* who, const uint32_t* bits_u, const uint32_t* bits_v, const float* h,
                        const float* l, const float* g, const float* x, const float* dy, const float* a_save,
                        const float* c_save, float* dx, float* dh, float* dl, float* dg, int64_t T, int64_t d_in,
                        int64_t d_out, int64_t r, float gscale, int accumulate, cudaStream_t st) {
    const int iT = (int)T, din = (int)d_in, dout = (int)d_out, ir = (int)r;
    const int BN = blr_bn(iT);
    const int ttiles = (iT + BN - 1) / BN, chunks = (iT + FIN_TC - 1) / FIN_TC;
    // column-sum partials of dh, dl and dg each in their own buffer, so that one
    // launch at the end finishes all three
    const int dh_parts = c_save ? chunks : ttiles;
    const size_t bytes = (size_t)T * r * 2 + 256 + ((size_t)dh_parts * d_out + 256) * 4 +
                         ((size_t)chunks * r + 256) * 4 + ((size_t)ttiles * d_in + 256) * 4 + 1024;
    void* mem = nullptr;
    cudaError_t e = cudaMallocAsync(&mem, bytes, st);
    if (e != cudaSuccess) return cuda_status(e, who);
    Scratch sc{reinterpret_cast<char*>(mem), 0};
    uint16_t* r16 = sc.take<uint16_t>((size_t)T * r);         // a.l (dh recompute), then b.l.gs
    float* colp_h = sc.take<float>((size_t)dh_parts * d_out);
    float* colp_l = sc.take<float>((size_t)chunks * r);
    float* colp_g = sc.take<float>((size_t)ttiles * d_in);
    const float inv_gs = 1.0f / gscale;

    // dh += sum_t dy.c
    if (c_save) {
        e = launch_pdl(colsum_prod_kernel, dim3((unsigned)((dout + 31) / 32), (unsigned)chunks), dim3(32, 8), 0, st,
                       dy, c_save, iT, dout, colp_h);
    } else {                                                 // recompute c = (a.l) S_U^T in the GEMM
        e = stage32(a_save, l, 1.0f, r16, iT, ir, st);
        if (e == cudaSuccess) {
            PlaneMaps pm;
            EpiArgs ep{nullptr, nullptr, nullptr, dy, colp_h, (int64_t)d_out, 1.0f};
            e = plane_maps_sign(pm, bits_u, dout, ir)
                    ? launch_umma<DecSign, EPI_COLSUM>(pm, ep, r16, iT, dout, ir, BN, 1, st)
                    : cudaErrorInvalidValue;
        }
    }
    // b = (dy.h.gs) S_U / gs in one pass over dy; dl += sum_t a.b; stage f16(b.l.gs)
    if (e == cudaSuccess)
        e = launch_blr_rank(dy, h, gscale, bits_u, iT, dout, ir, inv_gs, nullptr, l, gscale, r16, a_save, colp_l, st);
    // dx' = (b.l.gs) S_V / gs; dx = g.dx'; dg += sum_t x.dx'
    if (e == cudaSuccess) {
        PlaneMaps pm;
        EpiArgs ep{dx, nullptr, g, x, colp_g, (int64_t)d_in, inv_gs, accumulate};
        e = plane_maps_sign(pm, bits_v, din, ir)
                ? launch_umma<DecSign, EPI_SCALE_COLSUM>(pm, ep, r16, iT, din, ir, BN, 1, st)
                : cudaErrorInvalidValue;
    }
    // dh, dl, dg += their column sums, one launch
    if (e == cudaSuccess) {
        ColsumJobs jobs{{colp_h, colp_l, colp_g}, {dh_parts, chunks, ttiles}, {dout, ir, din}, {dh, dl, dg}};
        const int mxn = din > dout ? (din > ir ? din : ir) : (dout > ir ? dout : ir);
        e = launch_pdl(colsum_finish3_kernel, dim3((unsigned)((mxn + 255) / 256), 3u), dim3(256), 0, st, jobs);
    }
    cudaError_t e2 = cudaFreeAsync(mem, st);
    if (e != cudaSuccess) return cuda_status(e, who);
    return cuda_status(e2, who);
}


bool gscale_ok(float gscale) {
    int ex = 0;
    return gscale > 0.f && std::isfinite(gscale) && std::frexp(gscale, &ex) == 0.5f;
}

}  // namespace

extern "C" {

tq2_status blr_forward(const uint32_t* bits_u, const uint32_t* bits_v, const float* h, const float* l, const float* g,
                       const float* x, float* y, float* a_save, float* c_save, int64_t T, int64_t d_in, int64_t d_out,
                       int64_t r, void* stream) {
    if (!bits_u || !bits_v || !h || !l || !g || !x || !y || !a_save)
        return blr_fail(TQ2_EINVAL, "blr_forward: null pointer");
    tq2_status s = check_shapes("blr_forward", T, d_in, d_out, r);
    if (s != TQ2_OK) return s;
    if (!aligned16(x) || !aligned16(g) || !aligned16(l))
        return blr_fail(TQ2_EINVAL, "blr_forward: x, g and l must be 16-byte aligned");
    return forward_one("blr_forward", bits_u, bits_v, h, l, g, x, y, a_save, c_save, T, d_in, d_out, r, 0,
                       reinterpret_cast<cudaStream_t>(stream));
}

tq2_status blr_backward(const uint32_t* bits_u, const uint32_t* bits_v, const float* h, const float* l, const float* g,
                        const float* x, const float* dy, const float* a_save, const float* c_save, float* dx, float* dh,
                        float* dl, float* dg, int64_t T, int64_t d_in, int64_t d_out, int64_t r, float gscale,
                        void* stream) {
    if (!bits_u || !bits_v || !h || !l || !g || !x || !dy || !a_save || !dx || !dh || !dl || !dg)
        return blr_fail(TQ2_EINVAL, "blr_backward: null pointer");
    tq2_status s = check_shapes("blr_backward", T, d_in, d_out, r);
    if (s != TQ2_OK) return s;
    if (!gscale_ok(gscale)) return blr_fail(TQ2_EINVAL, "blr_backward: gscale must be a positive power of two");
    if (!aligned16(dy) || !aligned16(h) || !aligned16(l) || !aligned16(a_save))
        return blr_fail(TQ2_EINVAL, "blr_backward: dy, h, l and a_save must be 16-byte aligned");
    return backward_one("blr_backward", bits_u, bits_v, h, l, g, x, dy, a_save, c_save, dx, dh, dl, dg, T, d_in, d_out,
                        r, gscale, 0, reinterpret_cast<cudaStream_t>(stream));
}

tq2_status blr_forward_paths(const blr_path* paths, int P, const float* x, float* y, int64_t T, int64_t d_in,
                             int64_t d_out, int64_t r, void* stream) {
    if (!paths || !x || !y) return blr_fail(TQ2_EINVAL, "blr_forward_paths: null pointer");
    if (P < 1 || P > BLR_MAX_PATHS)
        return (tq2_status)set_error(TQ2_EINVAL, "blr_forward_paths: need 1 <= P <= 64 (P=%d)", P);
    tq2_status s = check_shapes("blr_forward_paths", T, d_in, d_out, r);
    if (s != TQ2_OK) return s;
    if (!aligned16(x)) return blr_fail(TQ2_EINVAL, "blr_forward_paths: x must be 16-byte aligned");
    for (int p = 0; p < P; ++p) {
        const blr_path& q = paths[p];
        if (!q.bits_u || !q.bits_v || !q.h || !q.l || !q.g || !q.a_save)
            return (tq2_status)set_error(TQ2_EINVAL, "blr_forward_paths: null pointer in path %d", p);
        if (!aligned16(q.g) || !aligned16(q.l))
            return (tq2_status)set_error(TQ2_EINVAL, "blr_forward_paths: g and l of path %d must be 16-byte aligned",
                                         p);
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    for (int p = 0; p < P; ++p) {
        const blr_path& q = paths[p];
        s = forward_one("blr_forward_paths", q.bits_u, q.bits_v, q.h, q.l, q.g, x, y, q.a_save, q.c_save, T, d_in,
                        d_out, r, p > 0 ? 1 : 0, st);
        if (s != TQ2_OK) return s;
    }
    return TQ2_OK;
}

tq2_status blr_backward_paths(const blr_path* paths, int P, const float* x, const float* dy, float* dx, int64_t T,
                              int64_t d_in, int64_t d_out, int64_t r, float gscale, void* stream) {
    if (!paths || !x || !dy || !dx) return blr_fail(TQ2_EINVAL, "blr_backward_paths: null pointer");
    if (P < 1 || P > BLR_MAX_PATHS)
        return (tq2_status)set_error(TQ2_EINVAL, "blr_backward_paths: need 1 <= P <= 64 (P=%d)", P);
    tq2_status s = check_shapes("blr_backward_paths", T, d_in, d_out, r);
    if (s != TQ2_OK) return s;
    if (!gscale_ok(gscale)) return blr_fail(TQ2_EINVAL, "blr_backward_paths: gscale must be a positive power of two");
    if (!aligned16(dy)) return blr_fail(TQ2_EINVAL, "blr_backward_paths: dy must be 16-byte aligned");
    for (int p = 0; p < P; ++p) {
        const blr_path& q = paths[p];
        if (!q.bits_u || !q.bits_v || !q.h || !q.l || !q.g || !q.a_save || !q.dh || !q.dl || !q.dg)
            return (tq2_status)set_error(TQ2_EINVAL, "blr_backward_paths: null pointer in path %d", p);
        if (!aligned16(q.h) || !aligned16(q.l) || !aligned16(q.a_save))
            return (tq2_status)set_error(TQ2_EINVAL,
                                         "blr_backward_paths: h, l and a_save of path %d must be 16-byte aligned", p);
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    for (int p = 0; p < P; ++p) {
        const blr_path& q = paths[p];
        s = backward_one("blr_backward_paths", q.bits_u, q.bits_v, q.h, q.l, q.g, x, dy, q.a_save, q.c_save, dx, q.dh,
                         q.dl, q.dg, T, d_in, d_out, r, gscale, p > 0 ? 1 : 0, st);
        if (s != TQ2_OK) return s;
    }
    return TQ2_OK;
}

tq2_status blr_sign_grads(const uint32_t* bits_u, const float* h, const float* l, const float* g, const float* x,
                          const float* dy, const float* a_save, float* gu, float* gv, int64_t T, int64_t d_in,
                          int64_t d_out, int64_t r, float gscale, void* stream) {
    if (!bits_u || !h || !l || !g || !x || !dy || !a_save || !gu || !gv)
        return blr_fail(TQ2_EINVAL, "blr_sign_grads: null pointer");
    tq2_status s = check_shapes("blr_sign_grads", T, d_in, d_out, r);
    if (s != TQ2_OK) return s;
    if (!gscale_ok(gscale)) return blr_fail(TQ2_EINVAL, "blr_sign_grads: gscale must be a positive power of two");
    if (!aligned16(dy) || !aligned16(h) || !aligned16(l) || !aligned16(g) || !aligned16(x) || !aligned16(a_save))
        return blr_fail(TQ2_EINVAL, "blr_sign_grads: x, dy, a_save, h, l and g must be 16-byte aligned");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int iT = (int)T, din = (int)d_in, dout = (int)d_out, ir = (int)r;
    const int Tp = (iT + 63) / 64 * 64;
    const int64_t mx = d_in > d_out ? d_in : d_out;
    const size_t bytes = (size_t)T * r * 4 + 256 + (size_t)T * r * 2 + 256 + (size_t)(mx + r) * Tp * 2 + 512;
    void* mem = nullptr;
    cudaError_t e = cudaMallocAsync(&mem, bytes, st);
    if (e != cudaSuccess) return cuda_status(e, "blr_sign_grads: scratch");
    Scratch sc{reinterpret_cast<char*>(mem), 0};
    float* b32 = sc.take<float>((size_t)T * r);
    uint16_t* b16 = sc.take<uint16_t>((size_t)T * r);      // the rank kernel's f16 staging (unused here)
    uint16_t* big = sc.take<uint16_t>((size_t)mx * Tp);     // (dy.h.gs)^T, then (x.g)^T
    uint16_t* small = sc.take<uint16_t>((size_t)r * Tp);    // (a.l)^T, then (b.l.gs)^T
    const float inv_gs = 1.0f / gscale;
    auto stage_t = [&](const float* src, int C, const float* col, float scale, uint16_t* dst) {
        return launch_pdl(stage_t16_kernel, dim3((unsigned)(C / 64), (unsigned)(Tp / 64)), dim3(256), 0, st, src, iT,
                          C, col, scale, dst, Tp);
    };
    // G[o][k] = (1/gs) sum_t rowsT[o][t] colsT[k][t]: A = colsT (r rows, DecDense), B = rowsT
    // (o tokens, TMA); the core writes out[token][row] = G[o][k].  Two K splits (atomic
    // add into a zeroed G, order-independent for two) when one split leaves SMs idle.
    auto gemm = [&](const uint16_t* colsT, const uint16_t* rowsT, int nrows, float* G) -> cudaError_t {
        int dev = 0, sms = 148;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int bn = umma_pick_bn(nrows);
        const int tiles = ((ir + UM_BM - 1) / UM_BM) * ((nrows + bn - 1) / bn);
        PlaneMaps pm;
        if (!plane_maps_dense(pm, colsT, ir, Tp)) return cudaErrorInvalidValue;
        EpiArgs ep{G, nullptr, nullptr, nullptr, nullptr, (int64_t)r, inv_gs};
        if (tiles < sms && Tp >= 2 * UM_BK) {
            cudaError_t e1 = cudaMemsetAsync(G, 0, (size_t)nrows * r * sizeof(float), st);
            if (e1 != cudaSuccess) return e1;
            return launch_umma<DecDense, EPI_ATOMIC>(pm, ep, rowsT, nrows, ir, Tp, bn, 2, st);
        }
        return launch_umma<DecDense, EPI_STORE>(pm, ep, rowsT, nrows, ir, Tp, bn, 1, st);
    };
    // b = (dy.h.gs) S_U / gs, as in the backward
    e = launch_blr_rank(dy, h, gscale, bits_u, iT, dout, ir, inv_gs, b32, l, gscale, b16, nullptr, nullptr, st);
    // G_U = diag(h) dy^T a diag(l), from (dy.h.gs)^T and (a.l)^T
    if (e == cudaSuccess) e = stage_t(dy, dout, h, gscale, big);
    if (e == cudaSuccess) e = stage_t(a_save, ir, l, 1.0f, small);
    if (e == cudaSuccess) e = gemm(small, big, dout, gu);
    // G_V = diag(g) x^T b diag(l), from (x.g)^T and (b.l.gs)^T
    if (e == cudaSuccess) e = stage_t(x, din, g, 1.0f, big);
    if (e == cudaSuccess) e = stage_t(b32, ir, l, gscale, small);
    if (e == cudaSuccess) e = gemm(small, big, din, gv);
    cudaError_t e2 = cudaFreeAsync(mem, st);
    if (e != cudaSuccess) return cuda_status(e, "blr_sign_grads");
    return cuda_status(e2, "blr_sign_grads: scratch free");
}

}  // extern "C"
