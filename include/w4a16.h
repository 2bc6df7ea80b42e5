/*
 * w4a16.h -- C ABI of libw4a16.so: fp16-activation x int4-weight group-quantized
 * GEMM for NVIDIA GB300 (sm_103a).
 *
 * Operation (github.com/justinchuby/onnx-genai pull 960, "What's landed" and
 * "Validation": fp16 x int4 MatMulNBits with per-group scales, group sizes
 * 16/32/64/128 and optional asymmetric 4-bit zero points):
 *
 *     Y[M,N] = A[M,K] . W[N,K]^T,   W[n,k] = (q[n,k] - zp[n,k/group]) * scale[n,k/group]
 *
 * Input formats (the plain reading of the "ONNX-native asymmetric-zp / nibble
 * format" named there):
 *   A       fp16 (IEEE binary16 bit patterns), row-major [M][K]
 *   q       uint8 [N][K/2]: nibble k of row n is byte k/2, low nibble for even k
 *   scales  fp16 or fp32, row-major [N][G], G = K/group
 *   zp      uint8 [N][ceil(G/2)], nibble j of row n = zero point of group j (low
 *           nibble for even j); NULL means symmetric (zero point 8)
 *   Y       fp16, row-major [M][N]; fp32 accumulation, round-to-nearest-even store
 *
 * Conventions shared by every call:
 *   - Device pointers are caller-owned device memory; host pointers are marked.
 *     The library never allocates, frees or synchronises inside a compute call;
 *     work is enqueued on `stream` (a cudaStream_t passed as void*, NULL = legacy
 *     default stream) and runs asynchronously.
 *   - Arguments are validated on the host before anything is launched; a
 *     non-OK status means nothing was enqueued. Launch failures map to
 *     W4A16_ERR_CUDA. No call throws.
 *   - Shape rules for the repacked layout and the kernels: M, N, K > 0,
 *     N % 16 == 0, K % 64 == 0, group in {16, 32, 64, 128}, K % group == 0.
 *     A, q_rep and Y must be 16-byte aligned, scales aligned to their element
 *     size. Violations return W4A16_ERR_INVALID_ARG or W4A16_ERR_UNSUPPORTED.
 *   - Results are deterministic: the same inputs and the same split factor give
 *     bit-identical Y on every run (fixed-order reductions, no atomics on data).
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W4A16_OK = 0,
    W4A16_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misalignment */
    W4A16_ERR_UNSUPPORTED = 2,   /* valid but outside the supported shape rules */
    W4A16_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
    W4A16_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    W4A16_ERR_TIMEOUT = 5        /* a bounded device-side wait expired */
} w4a16_status;

typedef enum { W4A16_SCALE_F16 = 0, W4A16_SCALE_F32 = 1 } w4a16_scale_dtype;

/* Which kernel family a GEMM call runs (reported by w4a16_gemm_plan). */
typedef enum {
    W4A16_PATH_SMALL_M = 0,      /* register-fed stream kernel, split-K over a cluster */
    W4A16_PATH_TCGEN05 = 1       /* TMA + tcgen05 tensor-memory kernel */
} w4a16_path;

/* Human-readable name of a status code (static storage, never NULL). */
const char *w4a16_status_string(w4a16_status s);

/* Bytes of the repacked weight buffer for an N x K int4 matrix: N*K/2. */
size_t w4a16_repacked_bytes(int N, int K);

/*
 * Repack nibble-packed int4 weights into the fragment-interleaved layout the GEMM
 * kernels read (the MatMulNBits pull request's "bijective ... reorder for
 * coalesced loads" with a device repack byte-identical to a host reference; the
 * permutation itself is this library's own):
 *   16-row sub-tile S = n/16, k-block b = k/64: piece (S, b) is 512 bytes at
 *   (S*(K/64) + b)*512, so every sub-tile is one contiguous run along K and a run
 *   of k-blocks of consecutive sub-tiles is a regular 3-D box for TMA copies;
 *   with g = n%8 and t = (k%16)/4 the 16-byte lane slot 4*g + (t + g/2)%4 of the
 *   piece at slot*16; u32 word j = (k%64)/16 at j*4; nibble p = 4*(e%2) + 2*(e/2)
 *   + h with e = k%4 and h = (n%16)/8 (byte p/2 of the word, high nibble when p
 *   is odd). Each lane slot holds one mma.sync m16n8k16 A fragment per word
 *   (rows g and g+8).
 *   q      device, uint8 [N][K/2] (input format above); not modified
 *   q_rep  device, w4a16_repacked_bytes(N, K) bytes, written; must not overlap q
 * Integer-only and bit-exact; inverse: w4a16_unpack_host.
 */
w4a16_status w4a16_repack(const uint8_t *q, uint8_t *q_rep, int N, int K, void *stream);

/*
 * Host inverse of w4a16_repack: q_rep (host, N*K/2 bytes) -> q (host, [N][K/2]).
 * Synchronous, pure host code, no CUDA calls.
 */
w4a16_status w4a16_unpack_host(const uint8_t *q_rep, uint8_t *q, int N, int K);

/*
 * Scratch bytes a w4a16_gemm call needs (0: split-K partials are reduced through
 * distributed shared memory inside a thread-block cluster, not global memory).
 * split_k: 0 = automatic, 1..8 = forced factor (small-M path).
 */
size_t w4a16_gemm_workspace_bytes(int M, int N, int K, int group, int split_k);

/*
 * Which path and split factor w4a16_gemm would use. split_k as in w4a16_gemm.
 * path / split_out are host pointers (either may be NULL).
 * Path choice: M above the small-M limit (w4a16_set_tuning, default 64) takes
 * the tensor-core path; so does M >= 33 (plain and fused SwiGLU) when that path's
 * grid (N/128 tiles, or N/64 for SwiGLU, times the token tiles) covers at least
 * two thirds of the SMs, unless split_k > 0 forces the small-M path's K split.
 * (This function reports the plain GEMM's choice.)
 */
w4a16_status w4a16_gemm_plan(int M, int N, int K, int group, int split_k,
                             int *path, int *split_out);

/*
 * Launch shape of the kernel a call would run: w4a16_gemm (swiglu_fused = 0) or
 * fused w4a16_gemm_swiglu (swiglu_fused = 1). For reports and tests; nothing is
 * launched. `info` is a host pointer. Errors as w4a16_gemm_plan.
 */
typedef struct {
    int path;          /* w4a16_path */
    int split;         /* CTAs along K per weight set (1 on the tensor-core path) */
    int ctas;          /* CTAs of the launch */
    int threads;       /* threads per CTA */
    int smem_bytes;    /* dynamic shared memory per CTA */
    int stages;        /* shared-memory ring stages of the weight stream */
} w4a16_launch_info;
w4a16_status w4a16_gemm_launch_info(int M, int N, int K, int group, int split_k, int swiglu_fused,
                                    w4a16_launch_info *info);

/*
 * Y = A . dequant(q_rep)^T  (see the operation at the top of this file).
 *   A        device fp16 [M][K], 16-byte aligned
 *   q_rep    device, repacked weights from w4a16_repack (N x K)
 *   scales   device [N][K/group], dtype sdt
 *   zp       device uint8 [N][ceil(G/2)] packed zero points, or NULL (zero point 8)
 *   Y        device fp16 [M][N], written (no read-modify-write)
 *   split_k  0 = automatic; 1..8 forces the small-M path's K split (a cluster
 *            of that many CTAs along K per run of sub-tiles) for M up to the
 *            small-M limit; ignored on the tensor-core path
 *   ws, ws_bytes  caller scratch of at least w4a16_gemm_workspace_bytes(); may be
 *            NULL when that is 0
 * Small M (see w4a16_gemm_plan for the choice) runs the stream kernel: weight
 * and activation boxes streamed by TMA through a shared-memory ring, each CTA a
 * run of 16-row sub-tiles over a K range, dequantisation in registers,
 * mma.sync m16n8k16 with fp32 accumulation and the group scale applied after
 * each group's partial sum (the pull request's "per-group scale AFTER the
 * tensor-core accumulate"); when the row split alone cannot fill the GPU, K is
 * split across a cluster and reduced in a fixed order.
 * Larger M runs the tcgen05 kernel: TMA-staged activations, int4 tiles dequantised to fp16
 * ((q - zp) * scale rounded once; fp32 scales are rounded to fp16 first) into
 * tensor memory, fp32 accumulation in tensor memory.
 */
w4a16_status w4a16_gemm(const uint16_t *A, const uint8_t *q_rep, const void *scales,
                        w4a16_scale_dtype sdt, const uint8_t *zp, uint16_t *Y,
                        int M, int N, int K, int group, int split_k,
                        void *ws, size_t ws_bytes, void *stream);

/*
 * w4a16_gemm for a caller whose activations arrive and whose outputs leave in
 * host memory (the same operation, defined at the top of this file): enqueues on
 * `stream` the copy of A_host into A_dev, the GEMM into Y_dev and the copy of
 * Y_dev into Y_host, one cudaMemcpyAsync per copy, and returns without
 * synchronising; Y_host holds the result once the stream has passed the call.
 *   A_host   host fp16 [M][K], page-locked (cudaHostAlloc, cudaHostRegister or
 *            torch pin_memory); not checked: with pageable memory the CUDA
 *            runtime performs the copies synchronously
 *   A_dev    device fp16 [M][K], 16-byte aligned, overwritten with A_host
 *   Y_dev    device fp16 [M][N], 16-byte aligned, overwritten with Y
 *   Y_host   host fp16 [M][N], page-locked as A_host, overwritten with Y
 *   q_rep, scales, sdt, zp, group, split_k as in w4a16_gemm (no workspace)
 * Every argument is validated before anything is enqueued, with the errors of
 * w4a16_gemm; a CUDA failure after the first copy was enqueued returns
 * W4A16_ERR_CUDA and may leave that copy enqueued.
 */
w4a16_status w4a16_gemm_host_io(const uint16_t *A_host, uint16_t *A_dev, const uint8_t *q_rep,
                                const void *scales, w4a16_scale_dtype sdt, const uint8_t *zp,
                                uint16_t *Y_dev, uint16_t *Y_host, int M, int N, int K, int group,
                                int split_k, void *stream);

/*
 * Scratch bytes for w4a16_gemm_swiglu: 0 when fused; 4*M*N (+alignment) when
 * unfused (the fp16 gate and up projections are materialised).
 */
size_t w4a16_swiglu_workspace_bytes(int M, int N, int K, int group, int fused);

/*
 * Y = silu(A . Wg^T) * (A . Wu^T), silu(x) = x / (1 + exp(-x)) (the pull
 * request's gate_up SwiGLU MLP fusion: paired gate/up int4 GEMMs followed by a
 * SiluMul epilogue). Gate and up share A, K, N, group and the scale dtype.
 *   fused = 1  one pass: both accumulators kept in fp32, silu*mul in the
 *              epilogue, only Y is written
 *   fused = 0  the unfused chain: gate -> fp16 G, up -> fp16 U (both in ws),
 *              then an elementwise silu_mul(G, U) -> Y
 * The two modes come from one source with this switch, for fusion benchmarks.
 */
w4a16_status w4a16_gemm_swiglu(const uint16_t *A,
                               const uint8_t *qg_rep, const void *sg, const uint8_t *zg,
                               const uint8_t *qu_rep, const void *su, const uint8_t *zu,
                               w4a16_scale_dtype sdt, uint16_t *Y,
                               int M, int N, int K, int group, int fused,
                               void *ws, size_t ws_bytes, void *stream);

/*
 * RMS-norm prologue (the pull request's "Update -- fused RMS-norm epilogue + e2e
 * PASS" and "Update -- P1 COMPLETE": the normalised activation is staged in
 * scratch, then the GEMM runs on it; gate_up SwiGLU has the same optional
 * prologue). The pages give no formula; the reading taken is the ONNX
 * SimplifiedLayerNormalization that the prologue replaces:
 *     An[m,k] = A[m,k] / sqrt(mean_k A[m,k]^2 + eps) * gamma[k]
 * computed in fp32 per row (fixed-order sum of squares) and stored as fp16 in
 * the caller's workspace; the GEMM (or SwiGLU) then runs on An exactly as
 * w4a16_gemm (w4a16_gemm_swiglu) would. With launch overlap on, the GEMM is a
 * programmatic dependent of the prologue and streams weights while it runs.
 *   gamma    device fp16 [K], 16-byte aligned
 *   eps      >= 0 (finite)
 *   ws       device scratch of w4a16_rmsnorm_workspace_bytes(M, N, K, group,
 *            mode) bytes, 256-byte aligned; mode 0 = w4a16_gemm_rmsnorm,
 *            1 = fused SwiGLU, 2 = unfused SwiGLU (An followed by the unfused
 *            chain's intermediates). Too small -> W4A16_ERR_WORKSPACE.
 * Other arguments, layouts and errors as w4a16_gemm / w4a16_gemm_swiglu.
 */
size_t w4a16_rmsnorm_workspace_bytes(int M, int N, int K, int group, int mode);
w4a16_status w4a16_gemm_rmsnorm(const uint16_t *A, const uint16_t *gamma, float eps, const uint8_t *q_rep,
                                const void *scales, w4a16_scale_dtype sdt, const uint8_t *zp, uint16_t *Y,
                                int M, int N, int K, int group, int split_k, void *ws, size_t ws_bytes,
                                void *stream);
w4a16_status w4a16_gemm_swiglu_rmsnorm(const uint16_t *A, const uint16_t *gamma, float eps,
                                       const uint8_t *qg_rep, const void *sg, const uint8_t *zg,
                                       const uint8_t *qu_rep, const void *su, const uint8_t *zu,
                                       w4a16_scale_dtype sdt, uint16_t *Y, int M, int N, int K, int group,
                                       int fused, void *ws, size_t ws_bytes, void *stream);

/*
 * Unfused SwiGLU (as w4a16_gemm_swiglu with fused = 0) for callers that cannot
 * allocate device memory -- code inside another framework's memory pool, hot
 * paths where an allocation that may synchronise the device is not allowed, or
 * plug-ins that are handed only input and output buffers. No counterpart in the
 * MatMulNBits pull request; this is a library convenience.
 *   The fp16 gate and up intermediates (4*M*N bytes) live in a fixed array
 *   compiled into the library, w4a16_swiglu_static_scratch_bytes() = 8 MiB,
 *   one per GPU that loads the library, kept until the process exits. Shapes
 *   whose 4*M*N exceeds it return W4A16_ERR_WORKSPACE and launch nothing.
 *   The call allocates and frees nothing. Its first call on a device looks up the
 *   array's device address (a runtime query, no allocation); make that first
 *   call before any stream capture on that device.
 *   Every call on a device shares the array, which keeps the last call's
 *   intermediates: calls that can overlap on the GPU (different streams without
 *   ordering between them) race and must not be issued that way. Nothing in the
 *   array needs to start at zero.
 *   Arguments, layouts and errors otherwise as w4a16_gemm_swiglu.
 */
size_t w4a16_swiglu_static_scratch_bytes(void);
w4a16_status w4a16_gemm_swiglu_unfused_static(const uint16_t *A,
                                              const uint8_t *qg_rep, const void *sg, const uint8_t *zg,
                                              const uint8_t *qu_rep, const void *su, const uint8_t *zu,
                                              w4a16_scale_dtype sdt, uint16_t *Y,
                                              int M, int N, int K, int group, void *stream);

/*
 * Tuning knobs (process-wide, not thread-safe; for tests and benchmarks).
 *   smallm_max  largest M that may take the small-M path (0 = default 64, max 64;
 *               -1 routes every M to the tensor-core path); see w4a16_gemm_plan
 */
w4a16_status w4a16_set_tuning(int smallm_max);

/*
 * Overlap of consecutive small-M GEMM calls (process-wide, not thread-safe;
 * default 0 = off). With enable = 1 each small-M launch is a programmatic
 * dependent of the work before it on the stream: its CTAs may start while that
 * work finishes, stage scales and zero points and start streaming q_rep, and
 * wait for it to complete before they read A or write Y. So A and Y may be the
 * previous call's output or input, as in a chain of layers, but q_rep, scales
 * and zp must not be written by the work that directly precedes the call on
 * the stream (weights loaded once and reused satisfy this; a w4a16_repack
 * followed at once by a GEMM on the same weights does not). Results are
 * identical with the switch on or off. The pages describe no such launch mode;
 * it is a GB300 launch-latency measure.
 * Returns W4A16_ERR_INVALID_ARG unless enable is 0 or 1.
 */
w4a16_status w4a16_set_launch_overlap(int enable);

/*
 * Limit of every bounded device-side wait (process-wide, not thread-safe; for
 * tests of the failure path). Each wait for an mbarrier phase (a copy landing,
 * a pipeline slot freeing up, the accumulator completing) gives up once it has
 * waited limit_ns or longer: the kernel then records W4A16_ERR_TIMEOUT in the
 * device error word (see w4a16_device_error), stops issuing work, waits for the
 * copies and tensor-core operations it already issued (with a fixed limit of
 * 0.2 s), releases its tensor memory and returns; its output is undefined.
 * Default 2000000000 (2 s). 0 gives up at the first poll that finds a phase
 * incomplete, which makes any call whose copies are still in flight fail; this
 * exists so that tests can run the expiry path without a stuck barrier.
 * Always returns W4A16_OK.
 */
w4a16_status w4a16_set_wait_limit_ns(unsigned long long limit_ns);

/*
 * Read and clear the device-side error word that bounded waits set when they
 * expire (W4A16_ERR_TIMEOUT) on the device current for the calling thread.
 * Synchronises `stream`. Returns W4A16_OK when no kernel reported an error.
 */
w4a16_status w4a16_device_error(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
