/*
 * tq2.h -- C ABI of the packed low-bit weight GEMM library for GB300 (sm_103a).
 *
 * One operation sits under two consumers:
 *
 *     out[m,n] = sum_k x[m,k] * W[n,k]
 *
 *  1. W in the ternary block format BlockTQ2_0_g128
 *     ("oxibonsai-kernels 0.2.1, src/gpu_backend/metal_graph/tests_gemm_tq2.rs",
 *     test test_encode_gemm_tq2_matches_reference): each 128-wide block of a
 *     weight row holds 32 bytes of 2-bit codes, 4 per byte, least significant
 *     first, code c meaning c-1 in {-1,0,+1}, and one f16 scale d;
 *     W[n,k] = (c-1)*d.
 *  2. The binary low-rank layer blr
 *     ("cortiq-engine 0.8.43, src/gpu_wgpu/train_mm.rs", module doc,
 *     blr_forward, blr_backward): W = diag(h) S_U diag(l) S_V^T diag(g) with
 *     the +-1 factors S_U, S_V stored as 1-bit bitmaps.
 *
 * Conventions for every entry point
 *   - Every call returns a tq2_status; nothing aborts the process.  Argument
 *     and shape errors are detected on the host before anything is launched.
 *     tq2_last_error() gives a one-line message for the calling thread.
 *   - "stream" is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Compute calls are asynchronous on that stream unless stated.
 *   - "DEVICE" pointers are CUDA device memory owned by the caller (for
 *     instance torch tensors); "HOST" pointers are ordinary host memory.
 *   - All float data is IEEE binary32, row-major, densely packed.
 *   - Device-side waits inside the kernels are bounded (about one second);
 *     when one runs out the kernel records TQ2_ETIMEOUT and returns early.
 *     tq2_device_status() reports (and clears) that record.
 *   - Activations are staged to f16 on the GPU; entries must be finite with
 *     |v| < 65504 or the results are not finite.
 */
#ifndef TQ2_GB300_H
#define TQ2_GB300_H

#include <stdint.h>

#if defined(__GNUC__)
#define TQ2_API __attribute__((visibility("default")))
#else
#define TQ2_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TQ2_OK = 0,
    TQ2_EINVAL = 1,          /* null pointer or bad argument value            */
    TQ2_ESHAPE = 2,          /* sizes break a documented shape rule           */
    TQ2_ENOMEM = 3,          /* device or host allocation failed              */
    TQ2_ECUDA = 4,           /* a CUDA runtime/driver call failed             */
    TQ2_ETIMEOUT = 5,        /* a bounded device-side wait ran out            */
    TQ2_EUNSUPPORTED = 6     /* no kernel for this device or configuration    */
} tq2_status;

/* Opaque weight handle; the library owns the device planes behind it. */
typedef struct tq2_weight* tq2_handle;

/* Kernel selection for tq2_gemm_path (tests and benchmarks). */
typedef enum {
    TQ2_PATH_AUTO = 0,       /* M <= 16: skinny kernel; otherwise tensor path */
    TQ2_PATH_SKINNY = 1,     /* decode-in-register kernel, f32 activations, M <= 16 */
    TQ2_PATH_TENSOR = 2      /* tcgen05 kernel, activations staged to f16     */
} tq2_path;

/* Static string for a status code. */
TQ2_API const char* tq2_status_string(int status);

/* Message of the last failure on the calling thread ("" if none). */
TQ2_API const char* tq2_last_error(void);

/* Library build identification, e.g. "tq2-gb300 sm_103a". */
TQ2_API const char* tq2_version(void);

/*
 * Synchronize `stream`, then report and clear the device-side error record
 * (TQ2_ETIMEOUT if a bounded wait in any kernel ran out since the last call,
 * TQ2_ECUDA if the stream reports an error, else TQ2_OK).
 */
TQ2_API tq2_status tq2_device_status(void* stream);

/*
 * tq2_debug_wait_timeout -- test export for the error path above: launches
 * one thread that waits, with a bound of limit_ns, on a shared-memory
 * barrier that nothing completes.  When the bound runs out it records the
 * timeout exactly as the library's kernels do and returns, so the next
 * tq2_device_status on that stream reports TQ2_ETIMEOUT (and clears it)
 * while the context stays usable.  Nothing faults, traps or hangs.
 *   limit_ns  0 < limit_ns <= 1e9 (the kernels' own bound), else TQ2_EINVAL.
 *   stream    asynchronous on it.
 */
TQ2_API tq2_status tq2_debug_wait_timeout(uint64_t limit_ns, void* stream);

/* ------------------------------------------------------------------------ */
/* Ternary TQ2 weights                                                       */
/* ------------------------------------------------------------------------ */

/*
 * tq2_upload -- copy BlockTQ2_0_g128 blocks to the device and repack them.
 * Passage: the public SoA cache path get_or_upload_tq2_weight_soa(key, aos)
 * of test test_encode_gemm_tq2_matches_reference ("oxibonsai-kernels 0.2.1,
 * tests_gemm_tq2.rs").
 *
 *   aos     HOST, N*(K/128) blocks of 34 bytes, row-major (block kb of row n
 *           at index n*(K/128)+kb).  Block = { uint8 qs[32]; f16 d (little
 *           endian) }; code i of qs[j] (bits 2i..2i+1) is element 4j+i of
 *           the block.  The caller keeps ownership; the bytes are copied.
 *   N, K    weight rows and inner dimension; N >= 1, K >= 128, K % 128 == 0,
 *           N*K < 2^40.  Else TQ2_ESHAPE.
 *   out     receives the handle (set to NULL on failure).
 *   stream  used for the copy and the repack kernel; the call synchronizes
 *           it before returning, so `aos` may be freed afterwards.
 *
 * Device layout behind the handle ("SoA"): a code plane uint8[N][K/4]
 * holding each row's qs bytes in K order, and a scale plane uint16[N][K/128]
 * of f16 bits, each followed by a little zeroed padding.  The tensor-core
 * path (M > 8) reads two further copies made here: the codes stage-tiled
 * (uint8[ceil(N/128)][K/64][128][16], a 64-code stage of 128 rows
 * contiguous) and the scales block-major (uint16[K/128][ceil(N/128)*128]),
 * rows past N zero; so a handle holds about 2*N*K/4 + N*K/64 bytes.  Codes
 * are not validated: code 3 decodes as +2 (3-1).
 */
TQ2_API tq2_status tq2_upload(const void* aos, int64_t N, int64_t K, tq2_handle* out, void* stream);

/* Release the handle and its device memory (NULL is accepted).  The caller
 * must make sure no work that reads it is still pending. */
TQ2_API tq2_status tq2_free(tq2_handle h);

/* Shape of a handle. */
TQ2_API tq2_status tq2_shape(tq2_handle h, int64_t* N, int64_t* K);

/*
 * tq2_gemm -- out[m,n] = sum_k x[m,k] * W[n,k].
 * Passage: encode_gemm_tq2(&handle, &input, &mut out, m, n, k) and its CPU
 * reference ("oxibonsai-kernels 0.2.1, tests_gemm_tq2.rs",
 * test_encode_gemm_tq2_matches_reference: out is row-major [M][N]).
 *
 *   x       DEVICE float[M][K], row-major, 16-byte aligned.
 *   out     DEVICE float[M][N], row-major, overwritten.
 *   M       0 <= M <= 2^24 (M == 0 is a no-op returning TQ2_OK); on the
 *           tensor path also M*K < 2^31.  Else TQ2_ESHAPE.
 *   N, K    must equal the handle's shape, else TQ2_ESHAPE.
 *   stream  asynchronous on this stream.  Internal scratch (f16 copies of
 *           x) is taken from the stream-ordered allocator of the current
 *           device and released on the same stream.
 *
 * M <= 16 runs the skinny kernel: each f32 activation is carried as two f16
 * terms, hi = f16(x) and lo = f16(x - hi), whose sum differs from x by at
 * most about 2^-22 |x| (the weights are exact), with f32 accumulation:
 * |error| <= 2^-12 sum_k |x[m,k] W[n,k]| + 1e-7 per element, which is within
 * the pages' 1e-3 at K <= 4096 for unit-scale data.  For M <= 8 and
 * MT*K <= 32768, with MT = M rounded up to 1, 2, 4 or 8, it is a single
 * kernel with no scratch (the fused GEMV); that kernel decodes
 * codes with an offset that it removes per 128-block, so the rounding of a
 * block that holds a nonzero weight scales with that block's sum of |x|
 * (tested within the bound above on weights with 99 % zeros and x up to 256x
 * unit scale).  On every path a block whose codes are all 1 contributes
 * exactly 0, so an all-zero row gives exactly 0.
 * M > 16 runs the tensor-core kernel: activations rounded to f16
 * (nearest-even), weights exact in f16, f32 accumulation;
 * |error| <= 1e-2 * sum_k |x[m,k] W[n,k]|.
 */
TQ2_API tq2_status tq2_gemm(tq2_handle h, const float* x, float* out, int64_t M, int64_t N, int64_t K,
                    void* stream);

/* tq2_gemm with an explicit kernel choice (tq2_path).  TQ2_PATH_SKINNY
 * requires M <= 16 (else TQ2_ESHAPE). */
TQ2_API tq2_status tq2_gemm_path(tq2_handle h, const float* x, float* out, int64_t M, int64_t N, int64_t K,
                         int path, void* stream);

/*
 * tq2_gemm_tensor_tuned -- the tensor-core path of tq2_gemm with its tile
 * shape chosen by the caller (tuning sweeps; no counterpart on the pages).
 *
 *   bn      tokens per tile: 0 = the library's choice, else a multiple of 16
 *           in 16..256 (one that is not a multiple of 32 must be >= M), or
 *           384 when N > 128.
 *   splits  K splits: 0 = the library's choice, else 1..16 and <= K/64.  With
 *           more than one split the partial sums are added into the
 *           (zeroed) output with atomic adds: two splits give the same bits
 *           in either order, more than two may differ between runs by
 *           rounding (all within the tensor-path bound of tq2_gemm).
 *   Other arguments and errors as tq2_gemm on its tensor path; a bad bn or
 *   splits returns TQ2_EINVAL.
 */
TQ2_API tq2_status tq2_gemm_tensor_tuned(tq2_handle h, const float* x, float* out, int64_t M, int64_t N,
                                         int64_t K, int bn, int splits, void* stream);

/*
 * tq2_gemm_grouped -- G independent decode-shape GEMMs in one launch:
 * out_g[m,n] = sum_k x_g[m,k] * W_g[n,k] for g < G, each as tq2_gemm with
 * M <= 8 computes it (same kernel, same per-output arithmetic, so results
 * are bit-identical to G separate tq2_gemm calls).  One launch streams all
 * G weights, so independent projections that read the same activations
 * (or different ones) do not pay G kernel launches and G dependency waits.
 *
 *   hs      HOST array of G handles; all must have the same K.
 *   xs      HOST array of G DEVICE pointers, float[M][K] each, 16-byte aligned.
 *   outs    HOST array of G DEVICE pointers, float[M][N_g] each (overwritten).
 *   G       1..64;  1 <= M <= 8 with MT*K <= 32768, MT = M rounded up to
 *           1, 2, 4 or 8 (x is held in shared memory);  K the handles' K.
 *           Else TQ2_ESHAPE.
 *   stream  asynchronous; no scratch is allocated.
 */
TQ2_API tq2_status tq2_gemm_grouped(const tq2_handle* hs, const float* const* xs, float* const* outs, int G,
                                    int64_t M, int64_t K, void* stream);

/*
 * tq2_unpack -- rebuild the AoS bytes from the device planes (round trip of
 * tq2_upload).  aos_out: HOST buffer of N*(K/128)*34 bytes.  Synchronous.
 */
TQ2_API tq2_status tq2_unpack(tq2_handle h, void* aos_out, void* stream);

/*
 * tq2_dequant_f16 -- W[n,k] = (c-1)*d as f16 bits, exact (code x scale is
 * representable in f16; "oxibonsai-kernels 0.2.1, tests_gemm_tq2.rs", the
 * v10 parity test notes that f16 staging of code x scale is exact).
 *   w   DEVICE uint16[N][K], overwritten.  Debug / test export.
 */
TQ2_API tq2_status tq2_dequant_f16(tq2_handle h, uint16_t* w, void* stream);

/*
 * tq2_quantize -- the ternary producer: f32 weights -> BlockTQ2_0_g128 blocks.
 * Passage: the 2-bit FakeQuantize helpers of "rlx-mlx 0.2.13,
 * src/lower/helpers.rs" (fq_q_max gives q_max = 1 for 2 bits; the scale is
 * max|w| / q_max floored at 1e-12; the value is round(w / scale) clamped to
 * [-q_max, q_max]), applied per 128-element block of a row in f32:
 *   s = max(max|w|, 1e-12);  q = clamp(round_half_even(w / s), -1, 1);
 *   code = q + 1;  d = f16(s), nearest with ties to even.
 * The block granularity and the half-to-even rounding are readings: the page
 * reduces per channel or per tensor and stores no codes.
 *
 *   w        DEVICE float32[N][K], row-major, finite values (NaN or Inf give
 *            unspecified codes).  Read only.
 *   N, K     N >= 1, K >= 128, K % 128 == 0, N*K < 2^40.  Else TQ2_ESHAPE.
 *   aos_out  DEVICE, N*(K/128) blocks of 34 bytes in the tq2_upload layout
 *            (block kb of row n at index n*(K/128)+kb), overwritten.  Copy
 *            it to the host and pass it to tq2_upload to use the weights.
 *   stream   the launch is asynchronous on it.
 * Null pointers: TQ2_EINVAL.
 */
TQ2_API tq2_status tq2_quantize(const float* w, int64_t N, int64_t K, void* aos_out, void* stream);

/*
 * tq2_gemm_skinny_static -- the skinny GEMM (M <= 16) without any device
 * allocation.  The pages have no counterpart to this call; it exists for
 * callers that must not allocate while they run a GEMM: plugin or custom-op
 * interfaces that forbid allocation inside their enqueue call, serving
 * processes that reserve all device memory up front, and real-time loops in
 * which an allocator call could stall or fail.
 *
 *   Same arguments as tq2_gemm with 1 <= M <= 16; it runs the same kernel
 *   as tq2_gemm (the fused GEMV where that applies, which needs no scratch,
 *   else the staged skinny kernel), so its results equal tq2_gemm's bit for
 *   bit.
 *   The handle must live on the current device, else TQ2_EINVAL.
 *   Scratch (staged kernel only): a fixed 1 MiB device array inside the
 *   library (one per GPU that loads it, held until the process exits) holds
 *   the staged f16 fragments of x, ceil(M/4)*K*16 bytes; larger requests (for example K > 16384 at
 *   M = 16, K > 65536 at M <= 4) return TQ2_ESHAPE.  No cudaMalloc,
 *   cudaFree or stream-ordered allocation is made.
 *   The first call on a device looks up the array's device address on the
 *   current device (cudaGetSymbolAddress) and caches it for the life of the
 *   process; make that first call before any stream capture, and do not call
 *   this function on a device after resetting it (cudaDeviceReset).
 *   Every call shares the one array: calls whose work may overlap on the GPU
 *   (different streams, or different threads without ordering) race on it.
 *   Nothing in it needs clearing between calls: each call writes every byte
 *   it later reads.
 */
TQ2_API tq2_status tq2_gemm_skinny_static(tq2_handle h, const float* x, float* out, int64_t M, int64_t N,
                                          int64_t K, void* stream);

/* ------------------------------------------------------------------------ */
/* Binary low-rank layer (blr)                                               */
/* ------------------------------------------------------------------------ */

/*
 * blr_expand_bits -- sign bitmap to an f16 +-1 plane (bit-exact).
 * Passage: kernels expand_n / expand_t ("cortiq-engine 0.8.43,
 * train_mm.rs"): bitmap [rows][r/32] u32, bit j of word w is rank 32w+j,
 * a set bit is +1.0, a clear bit -1.0.
 *   bits       DEVICE uint32[rows][r/32].
 *   plane_f16  DEVICE uint16[rows][r] (transpose == 0) or [r][rows]
 *              (transpose != 0), f16 bits, overwritten.
 *   rows >= 1; r >= 32, r % 32 == 0.
 */
TQ2_API tq2_status blr_expand_bits(const uint32_t* bits, int64_t rows, int64_t r, uint16_t* plane_f16,
                           int transpose, void* stream);

/*
 * blr_forward -- one path of the binary low-rank layer, forward.
 * Passage: blr_forward and the module doc ("cortiq-engine 0.8.43,
 * train_mm.rs"):  a = (x.g) S_V,  c = (a.l) S_U^T,  y = h.c
 * (elementwise products broadcast over tokens).
 *
 *   bits_u  DEVICE uint32[d_out][r/32]  (S_U, [d_out][r])
 *   bits_v  DEVICE uint32[d_in][r/32]   (S_V, [d_in][r])
 *   h       DEVICE float[d_out];  l  DEVICE float[r];  g  DEVICE float[d_in]
 *   x       DEVICE float[T][d_in]
 *   y       DEVICE float[T][d_out], overwritten
 *   a_save  DEVICE float[T][r], overwritten with a (needed by blr_backward)
 *   c_save  DEVICE float[T][d_out] overwritten with c, or NULL (then
 *           blr_backward recomputes c from a_save)
 *   T >= 1; d_in, d_out multiples of 64; r >= 128, r % 128 == 0 (the page
 *   requires a multiple of 128); T*max(d_in, d_out) < 2^31, T*r < 2^28 and
 *   d_in, d_out <= 2^20.  Else TQ2_ESHAPE.  x, g and l must be 16-byte
 *   aligned (TQ2_EINVAL otherwise).
 * The activations x.g and a.l are staged to f16 (nearest-even); the GEMMs
 * accumulate in f32.  Scratch comes from the stream-ordered allocator.
 */
TQ2_API tq2_status blr_forward(const uint32_t* bits_u, const uint32_t* bits_v, const float* h,
                       const float* l, const float* g, const float* x, float* y,
                       float* a_save, float* c_save, int64_t T, int64_t d_in, int64_t d_out,
                       int64_t r, void* stream);

/*
 * blr_backward -- one path of the binary low-rank layer, backward.
 * Passage: blr_backward and the module doc ("cortiq-engine 0.8.43,
 * train_mm.rs"):
 *   dh += sum_t dy.c     b   = (dy.h) S_U     dl += sum_t a.b
 *   dx' = (b.l) S_V^T    dg += sum_t x.dx'    dx  = g.dx'
 *
 *   x, dy         DEVICE float[T][d_in], float[T][d_out]
 *   a_save        DEVICE float[T][r] from blr_forward on the same x
 *   c_save        DEVICE float[T][d_out] from blr_forward, or NULL (recompute)
 *   dx            DEVICE float[T][d_in], overwritten
 *   dh, dl, dg    DEVICE float[d_out], float[r], float[d_in]; ACCUMULATED
 *                 (+=) as on the page; the caller zeroes them.
 *   gscale        power of two (1.0 allowed) multiplying the gradients while
 *                 they are staged in f16, divided back out after each GEMM
 *                 (the page keeps gradients out of the f16 subnormals this
 *                 way).  Else TQ2_EINVAL.
 * Column sums use a fixed reduction order (deterministic run to run).
 * Shape rules as blr_forward; dy, h, l and a_save must be 16-byte aligned.
 */
TQ2_API tq2_status blr_backward(const uint32_t* bits_u, const uint32_t* bits_v, const float* h,
                        const float* l, const float* g, const float* x, const float* dy,
                        const float* a_save, const float* c_save, float* dx, float* dh,
                        float* dl, float* dg, int64_t T, int64_t d_in, int64_t d_out,
                        int64_t r, float gscale, void* stream);

/*
 * Several paths of one blr layer, y = sum_p diag(h_p) S_U,p diag(l_p) S_V,p^T
 * diag(g_p) x.  Passage: blr_forward / blr_backward over layer.paths and the
 * two-path combine scale_acc2 ("cortiq-engine 0.8.43, train_mm.rs"): the
 * paths are taken in order, the first writes y (dx) and each later one adds
 * its product to it, each product and each sum rounded to f32 separately
 * (no fused multiply-add): for two paths y = fl(fl(h0.c0) + fl(h1.c1)), the
 * page's one-pass two-path rounding; for more, fl(fl(y + fl(h_p.c_p))) in
 * path order, as the page's scale_acc passes.
 *
 * One path: its bitmaps and vectors (DEVICE, layouts as blr_forward), its
 * forward outputs a_save (required) and c_save (may be NULL), and its
 * gradient accumulators dh, dl, dg (DEVICE, += as in blr_backward; used by
 * blr_backward_paths only).
 */
typedef struct {
    const uint32_t* bits_u;
    const uint32_t* bits_v;
    const float* h;
    const float* l;
    const float* g;
    float* a_save;
    float* c_save;
    float* dh;
    float* dl;
    float* dg;
} blr_path;

#define BLR_MAX_PATHS 64

/*
 * blr_forward_paths -- forward of a layer of P paths (1 <= P <= BLR_MAX_PATHS).
 *   paths   HOST array of P blr_path (read during the call only).
 *   x       DEVICE float[T][d_in], shared by all paths.
 *   y       DEVICE float[T][d_out], overwritten with the combined output.
 * Shape rules as blr_forward.  x and each path's g and l must be 16-byte
 * aligned.  With P = 1 the result is blr_forward's bit for bit.
 */
TQ2_API tq2_status blr_forward_paths(const blr_path* paths, int P, const float* x, float* y, int64_t T,
                             int64_t d_in, int64_t d_out, int64_t r, void* stream);

/*
 * blr_backward_paths -- backward of the layer of the last blr_forward_paths
 * on the same x: each path's dh, dl, dg accumulate (+=), dx (DEVICE
 * float[T][d_in]) is overwritten with sum_p g_p.dx'_p rounded as described
 * above.  gscale as blr_backward; dy and each path's h, l and a_save must be
 * 16-byte aligned.
 */
TQ2_API tq2_status blr_backward_paths(const blr_path* paths, int P, const float* x, const float* dy, float* dx,
                              int64_t T, int64_t d_in, int64_t d_out, int64_t r, float gscale,
                              void* stream);

/*
 * blr_sign_grads -- the gradients of the loss with respect to one path's
 * signs, G_U = diag(h) dy^T a diag(l) ([d_out][r]) and
 * G_V = diag(g) x^T b diag(l) ([d_in][r]) with b = (dy.h) S_U.
 * Passage: blr_backward's sign-training step and the test
 * blr_sign_flip_exact ("cortiq-engine 0.8.43, train_mm.rs"): the token axis
 * is the GEMMs' K, the operands dy.h.gs, a.l, x.g and b.l.gs are staged
 * transposed in f16, and flipping sign s of U[i,k] changes L = 1/2|y - y*|^2
 * by -2 s G_U[i,k] + 2 h_i^2 l_k^2 sum_t a_tk^2 (V likewise).
 *
 *   bits_u        DEVICE uint32[d_out][r/32] (S_U; S_V is not needed)
 *   h, l, g       DEVICE float[d_out], float[r], float[d_in]
 *   x, dy         DEVICE float[T][d_in], float[T][d_out]
 *   a_save        DEVICE float[T][r] from blr_forward on the same x
 *   gu, gv        DEVICE float[d_out][r], float[d_in][r], overwritten
 *   gscale        power of two multiplying the dy-side operands while they
 *                 are staged in f16, divided back out (as blr_backward);
 *                 dy.h.gs and b.l.gs must stay inside the f16 range (a
 *                 value beyond 65504 stages as inf).
 * Shape rules as blr_forward; x, dy, a_save, h, l and g must be 16-byte
 * aligned (TQ2_EINVAL otherwise).
 */
TQ2_API tq2_status blr_sign_grads(const uint32_t* bits_u, const float* h, const float* l, const float* g,
                          const float* x, const float* dy, const float* a_save, float* gu, float* gv,
                          int64_t T, int64_t d_in, int64_t d_out, int64_t r, float gscale, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TQ2_GB300_H */
