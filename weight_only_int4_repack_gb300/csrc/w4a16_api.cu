// C ABI of libw4a16.so: argument validation, path and split planning, dispatch.
// Nothing here allocates, frees or synchronises on the compute calls; every
// check runs on the host before the first launch.
#include <climits>
#include <cstring>
#include <mutex>
#include <set>
#include <utility>

#include "w4a16_internal.h"

using namespace w4a16;

namespace {

int g_smallm_max = kSmallMMaxM;
int g_launch_overlap = 0;  // small-M launches as programmatic dependents
unsigned long long g_wait_ns = 2000000000ull;  // limit of every bounded device-side wait

__device__ unsigned int g_device_error;  // set by bounded waits that expire

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Per-device caches below are filled on first use under this lock, so that
// concurrent first calls from several host threads are well defined.
std::mutex g_cache_mu;

// Device address of the error word on the current device (looked up once per device).
unsigned int *device_error_ptr() {
    static unsigned int *cached[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_cache_mu);
    if (!cached[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess) return nullptr;
        cached[dev] = static_cast<unsigned int *>(ptr);
    }
    return cached[dev];
}

}  // namespace

cudaError_t w4a16::ensure_max_dyn_smem(const void *func, int bytes) {
    static std::set<std::pair<const void *, int>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_cache_mu);
    if (done.count({func, dev})) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.insert({func, dev});
    return e;
}

// Number of SMs of the current device (queried once per device).
int w4a16::sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(g_cache_mu);
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

namespace {

w4a16_status check_shape(int M, int N, int K, int group) {
    if (M <= 0 || N <= 0 || K <= 0) return W4A16_ERR_INVALID_ARG;
    if (group != 16 && group != 32 && group != 64 && group != 128) return W4A16_ERR_UNSUPPORTED;
    if (K % 2 != 0 || K % group != 0) return W4A16_ERR_INVALID_ARG;
    if (N % kSubRows != 0 || K % kKBlock != 0) return W4A16_ERR_UNSUPPORTED;
    // Index arithmetic uses 64-bit offsets; keep each dimension product sane.
    if ((long long)M * K > (1LL << 40) || (long long)N * K > (1LL << 40) ||
        (long long)M * N > (1LL << 40))
        return W4A16_ERR_UNSUPPORTED;
    return W4A16_OK;
}

w4a16_status check_weights(const uint8_t *q_rep, const void *scales, w4a16_scale_dtype sdt) {
    if (!q_rep || !scales) return W4A16_ERR_INVALID_ARG;
    if (sdt != W4A16_SCALE_F16 && sdt != W4A16_SCALE_F32) return W4A16_ERR_INVALID_ARG;
    if (!aligned(q_rep, 16)) return W4A16_ERR_INVALID_ARG;
    if (!aligned(scales, sdt == W4A16_SCALE_F32 ? 4 : 2)) return W4A16_ERR_INVALID_ARG;
    return W4A16_OK;
}

struct Plan {
    int path;
    SmallMPlan sm;  // small-M path only
};

// The tensor-core kernel costs nearly the same for any M up to its token tile,
// so from a few dozen tokens on it beats the stream kernel once its grid fills
// most SMs. Past 32 tokens the stream kernel works on eight 8-token tiles (its
// cost jumps), so both the plain GEMM and fused SwiGLU switch at 33 tokens.
// Measured on GB300 (us per call, stream kernel vs tensor-core kernel): K=5120
// N=13824 (108 tiles) M=32 29.2 vs 37.1, M=33 about 51 vs 37, M=40 49.3 vs 38.5,
// M=64 56.2 vs 38.6; K=N=4096 (32 tiles, too few for the tensor-core grid)
// M=64 15.8 vs 31.6. Fused SwiGLU at K=5120 N=13824: M=32 52.3 (stream, split 2)
// vs 73 (tensor core), M=33 126.9 vs 73.0.
constexpr int kTcMinM = 33;
constexpr int kTcMinMSwiglu = 33;
bool tc_preferred(int M, int N, bool swiglu) {
    if (M < (swiglu ? kTcMinMSwiglu : kTcMinM)) return false;
    const int cols = swiglu ? 64 : kTileRows;  // output columns per tensor-core CTA
    const int T = tc_tile_tokens(M, swiglu);
    const long long ctas = (long long)((N + cols - 1) / cols) * ((M + T - 1) / T);
    return 3 * ctas >= 2LL * sm_count();
}

w4a16_status make_plan(int M, int N, int K, int group, int split_k, bool swiglu, bool scale_f32, Plan *out) {
    if (split_k < 0 || split_k > 8) return W4A16_ERR_INVALID_ARG;
    Plan p{};
    const int smax = g_smallm_max;
    // A forced K split exists only on the small-M path, so it keeps that path.
    if (M <= smax && (split_k > 0 || !tc_preferred(M, N, swiglu))) {
        p.path = W4A16_PATH_SMALL_M;
        if (split_k > K / (group > kKBlock ? group : kKBlock)) return W4A16_ERR_UNSUPPORTED;
        (void)scale_f32;
        p.sm = smallm_plan(M, N, K, group, swiglu, split_k, sm_count());
        if (p.sm.split <= 0) return W4A16_ERR_UNSUPPORTED;
    } else {
        p.path = W4A16_PATH_TCGEN05;
        p.sm = SmallMPlan{1, 0, 0, 0};
    }
    *out = p;
    return W4A16_OK;
}

w4a16_status from_cuda(cudaError_t e) { return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------------------
// Unfused SwiGLU epilogue: Y = silu(G) * U on fp16 tensors, fp32 arithmetic.
// ---------------------------------------------------------------------------
__global__ void silu_mul_kernel(const uint4 *__restrict__ G, const uint4 *__restrict__ U,
                                uint4 *__restrict__ Y, size_t n_vec) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec;
         i += (size_t)gridDim.x * blockDim.x) {
        const uint4 gv = G[i], uv = U[i];
        uint4 yv;
        const __half2 *gh = reinterpret_cast<const __half2 *>(&gv);
        const __half2 *uh = reinterpret_cast<const __half2 *>(&uv);
        __half2 *yh = reinterpret_cast<__half2 *>(&yv);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 gf = __half22float2(gh[j]);
            const float2 uf = __half22float2(uh[j]);
            const float a = gf.x / (1.0f + expf(-gf.x)) * uf.x;
            const float b = gf.y / (1.0f + expf(-gf.y)) * uf.y;
            yh[j] = __floats2half2_rn(a, b);
        }
        Y[i] = yv;
    }
}

// ---------------------------------------------------------------------------
// RMS-norm prologue: An[m,k] = fp16(A[m,k] * r_m * gamma[k]),
// r_m = 1 / sqrt(mean_k A[m,k]^2 + eps), fp32 arithmetic. One CTA per row; the
// sum of squares is reduced in a fixed order (deterministic).
// ---------------------------------------------------------------------------
constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const uint4 *__restrict__ A, const uint4 *__restrict__ gamma,
                                                               uint4 *__restrict__ An, int K, float eps) {
    __shared__ float red[kNormThreads / 32];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");  // A may be the previous kernel's output
    const int nv = K / 8;
    const uint4 *row = A + (size_t)blockIdx.x * nv;
    float ss = 0.f;
    for (int i = threadIdx.x; i < nv; i += kNormThreads) {
        const uint4 x = row[i];
        const __half2 *h = reinterpret_cast<const __half2 *>(&x);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(h[e]);
            ss = fmaf(f.x, f.x, ss);
            ss = fmaf(f.y, f.y, ss);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) tot += red[w];
    const float r = 1.0f / sqrtf(tot / (float)K + eps);
    uint4 *out = An + (size_t)blockIdx.x * nv;
    for (int i = threadIdx.x; i < nv; i += kNormThreads) {
        const uint4 x = row[i], gv = gamma[i];
        const __half2 *h = reinterpret_cast<const __half2 *>(&x);
        const __half2 *gh = reinterpret_cast<const __half2 *>(&gv);
        uint4 y;
        __half2 *yh = reinterpret_cast<__half2 *>(&y);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(h[e]);
            const float2 gf = __half22float2(gh[e]);
            yh[e] = __floats2half2_rn(f.x * r * gf.x, f.y * r * gf.y);
        }
        out[i] = y;
    }
}

}  // namespace

namespace w4a16 {
cudaError_t launch_rmsnorm(const __half *A, const __half *gamma, __half *An, int M, int K, float eps, bool overlap,
                           cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)M, 1, 1);
    cfg.blockDim = dim3(kNormThreads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, rmsnorm_kernel, reinterpret_cast<const uint4 *>(A),
                              reinterpret_cast<const uint4 *>(gamma), reinterpret_cast<uint4 *>(An), K, eps);
}

cudaError_t launch_silu_mul(const __half *G, const __half *U, __half *Y, size_t n, cudaStream_t s) {
    const size_t n_vec = n / 8;  // n is a multiple of 8 (N % 16 == 0)
    const int threads = 256;
    size_t blocks = (n_vec + threads - 1) / threads;
    const size_t cap = (size_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    silu_mul_kernel<<<(unsigned)blocks, threads, 0, s>>>(reinterpret_cast<const uint4 *>(G),
                                                        reinterpret_cast<const uint4 *>(U),
                                                        reinterpret_cast<uint4 *>(Y), n_vec);
    return cudaGetLastError();
}
}  // namespace w4a16

extern "C" {

const char *w4a16_status_string(w4a16_status s) {
    switch (s) {
        case W4A16_OK: return "ok";
        case W4A16_ERR_INVALID_ARG: return "invalid argument";
        case W4A16_ERR_UNSUPPORTED: return "unsupported shape or configuration";
        case W4A16_ERR_WORKSPACE: return "workspace missing or too small";
        case W4A16_ERR_CUDA: return "CUDA error";
        case W4A16_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

size_t w4a16_repacked_bytes(int N, int K) {
    if (N <= 0 || K <= 0) return 0;
    return (size_t)N * (size_t)K / 2;
}

w4a16_status w4a16_repack(const uint8_t *q, uint8_t *q_rep, int N, int K, void *stream) {
    if (!q || !q_rep || N <= 0 || K <= 0) return W4A16_ERR_INVALID_ARG;
    if (N % kSubRows || K % kKBlock) return W4A16_ERR_UNSUPPORTED;
    if (!aligned(q, 2) || !aligned(q_rep, 16)) return W4A16_ERR_INVALID_ARG;
    const size_t bytes = (size_t)N * K / 2;
    const uintptr_t a = (uintptr_t)q, b = (uintptr_t)q_rep;
    if (a < b + bytes && b < a + bytes) return W4A16_ERR_INVALID_ARG;  // must not overlap
    return from_cuda(launch_repack(q, q_rep, N, K, (cudaStream_t)stream));
}

w4a16_status w4a16_unpack_host(const uint8_t *q_rep, uint8_t *q, int N, int K) {
    if (!q_rep || !q || N <= 0 || K <= 0) return W4A16_ERR_INVALID_ARG;
    if (N % kSubRows || K % kKBlock) return W4A16_ERR_UNSUPPORTED;
    const size_t row_bytes = (size_t)K / 2;
    const int kblocks = K / kKBlock;
    for (int S = 0; S < N / kSubRows; ++S) {
        for (int b = 0; b < kblocks; ++b) {
            const uint8_t *piece = q_rep + piece_offset(S, b, K);
            for (int slot = 0; slot < 32; ++slot) {
                const int g = slot / 4, t = ((slot % 4) - g / 2 + 4) % 4;
                for (int j = 0; j < 4; ++j) {
                    const uint8_t *wp = piece + slot * 16 + j * 4;
                    const uint32_t word = (uint32_t)wp[0] | ((uint32_t)wp[1] << 8) |
                                          ((uint32_t)wp[2] << 16) | ((uint32_t)wp[3] << 24);
                    for (int h = 0; h < 2; ++h) {
                        const int row = S * kSubRows + g + 8 * h;
                        for (int e = 0; e < 4; ++e) {
                            const int p = 4 * (e % 2) + 2 * (e / 2) + h;
                            const uint8_t nib = (uint8_t)((word >> (4 * p)) & 0xF);
                            const int k = b * kKBlock + 16 * j + 4 * t + e;
                            uint8_t &dst = q[(size_t)row * row_bytes + k / 2];
                            dst = (k % 2 == 0) ? (uint8_t)((dst & 0xF0) | nib)
                                               : (uint8_t)((dst & 0x0F) | (nib << 4));
                        }
                    }
                }
            }
        }
    }
    return W4A16_OK;
}

size_t w4a16_gemm_workspace_bytes(int M, int N, int K, int group, int split_k) {
    (void)M; (void)N; (void)K; (void)group; (void)split_k;
    return 0;
}

w4a16_status w4a16_gemm_plan(int M, int N, int K, int group, int split_k, int *path, int *split_out) {
    w4a16_status st = check_shape(M, N, K, group);
    if (st != W4A16_OK) return st;
    Plan p;
    st = make_plan(M, N, K, group, split_k, false, false, &p);
    if (st != W4A16_OK) return st;
    if (path) *path = p.path;
    if (split_out) *split_out = p.sm.split;
    return W4A16_OK;
}

w4a16_status w4a16_gemm_launch_info(int M, int N, int K, int group, int split_k, int swiglu_fused,
                                    w4a16_launch_info *info) {
    w4a16_status st = check_shape(M, N, K, group);
    if (st != W4A16_OK) return st;
    if (!info || (swiglu_fused != 0 && swiglu_fused != 1)) return W4A16_ERR_INVALID_ARG;
    const bool sw = swiglu_fused == 1;
    Plan p;
    if ((st = make_plan(M, N, K, group, sw ? 0 : split_k, sw, false, &p)) != W4A16_OK) return st;
    w4a16_launch_info r{};
    r.path = p.path;
    if (p.path == W4A16_PATH_TCGEN05) {
        r.split = 1;
        tc_launch_shape(M, N, sw, &r.ctas, &r.threads, &r.smem_bytes, &r.stages);
    } else {  // small-M tile kernel
        r.split = p.sm.split;
        r.ctas = ((N + kTileRows - 1) / kTileRows) * p.sm.split * (sw ? 2 : 1);
        r.threads = smallm_threads(M, sw);
        r.smem_bytes = p.sm.smem;
        r.stages = 2;
    }
    *info = r;
    return W4A16_OK;
}

static w4a16_status gemm_impl(const uint16_t *A, const WeightSet *ws_sets, int nsets,
                              w4a16_scale_dtype sdt, uint16_t *Y, int M, int N, int K, int group,
                              int split_k, cudaStream_t stream) {
    Plan plan;
    w4a16_status st = make_plan(M, N, K, group, split_k, nsets == 2, sdt == W4A16_SCALE_F32, &plan);
    if (st != W4A16_OK) return st;
    unsigned int *err = device_error_ptr();
    if (!err) return W4A16_ERR_CUDA;
    if (plan.path == W4A16_PATH_TCGEN05) {
        TcParams t{};
        t.A = reinterpret_cast<const __half *>(A);
        t.w[0] = ws_sets[0];
        t.w[1] = nsets == 2 ? ws_sets[1] : ws_sets[0];
        t.Y = reinterpret_cast<__half *>(Y);
        t.M = M; t.N = N; t.K = K; t.G = K / group;
        t.scale_f32 = sdt == W4A16_SCALE_F32;
        t.err = err;
        t.wait_ns = g_wait_ns;
        return from_cuda(launch_tc(t, group, nsets == 2, stream));
    }
    SmallMParams p{};
    p.A = reinterpret_cast<const __half *>(A);
    p.w[0] = ws_sets[0];
    p.w[1] = nsets == 2 ? ws_sets[1] : ws_sets[0];
    p.Y = reinterpret_cast<__half *>(Y);
    p.M = M; p.N = N; p.K = K; p.G = K / group;
    p.scale_f32 = sdt == W4A16_SCALE_F32;
    p.split = plan.sm.split;
    p.kc_blocks = plan.sm.kc;
    p.overlap = g_launch_overlap;
    p.err = err;
    p.wait_ns = g_wait_ns;
    return from_cuda(launch_smallm(p, group, nsets == 2, stream));
}

w4a16_status w4a16_gemm(const uint16_t *A, const uint8_t *q_rep, const void *scales,
                        w4a16_scale_dtype sdt, const uint8_t *zp, uint16_t *Y,
                        int M, int N, int K, int group, int split_k,
                        void *ws, size_t ws_bytes, void *stream) {
    (void)ws; (void)ws_bytes;
    w4a16_status st = check_shape(M, N, K, group);
    if (st != W4A16_OK) return st;
    if (!A || !Y) return W4A16_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(Y, 16)) return W4A16_ERR_INVALID_ARG;
    st = check_weights(q_rep, scales, sdt);
    if (st != W4A16_OK) return st;
    const WeightSet w{q_rep, scales, zp};
    return gemm_impl(A, &w, 1, sdt, Y, M, N, K, group, split_k, (cudaStream_t)stream);
}

w4a16_status w4a16_gemm_host_io(const uint16_t *A_host, uint16_t *A_dev, const uint8_t *q_rep,
                                const void *scales, w4a16_scale_dtype sdt, const uint8_t *zp,
                                uint16_t *Y_dev, uint16_t *Y_host, int M, int N, int K, int group,
                                int split_k, void *stream) {
    w4a16_status st = check_shape(M, N, K, group);
    if (st != W4A16_OK) return st;
    if (!A_host || !A_dev || !Y_dev || !Y_host) return W4A16_ERR_INVALID_ARG;
    if (!aligned(A_dev, 16) || !aligned(Y_dev, 16)) return W4A16_ERR_INVALID_ARG;
    if ((st = check_weights(q_rep, scales, sdt)) != W4A16_OK) return st;
    Plan plan;  // the plan's checks (split_k, shape) before the first copy is enqueued
    if ((st = make_plan(M, N, K, group, split_k, false, sdt == W4A16_SCALE_F32, &plan)) != W4A16_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    st = from_cuda(cudaMemcpyAsync(A_dev, A_host, (size_t)M * K * 2, cudaMemcpyHostToDevice, s));
    if (st != W4A16_OK) return st;
    const WeightSet w{q_rep, scales, zp};
    if ((st = gemm_impl(A_dev, &w, 1, sdt, Y_dev, M, N, K, group, split_k, s)) != W4A16_OK) return st;
    return from_cuda(cudaMemcpyAsync(Y_host, Y_dev, (size_t)M * N * 2, cudaMemcpyDeviceToHost, s));
}

size_t w4a16_swiglu_workspace_bytes(int M, int N, int K, int group, int fused) {
    (void)K; (void)group;
    if (fused || M <= 0 || N <= 0) return 0;
    return 2 * align_up((size_t)M * N * 2, 256);
}

w4a16_status w4a16_gemm_swiglu(const uint16_t *A,
                               const uint8_t *qg_rep, const void *sg, const uint8_t *zg,
                               const uint8_t *qu_rep, const void *su, const uint8_t *zu,
                               w4a16_scale_dtype sdt, uint16_t *Y,
                               int M, int N, int K, int group, int fused,
                               void *ws, size_t ws_bytes, void *stream) {
    w4a16_status st = check_shape(M, N, K, group);
    if (st != W4A16_OK) return st;
    if (!A || !Y) return W4A16_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(Y, 16)) return W4A16_ERR_INVALID_ARG;
    if ((st = check_weights(qg_rep, sg, sdt)) != W4A16_OK) return st;
    if ((st = check_weights(qu_rep, su, sdt)) != W4A16_OK) return st;
    const WeightSet sets[2] = {{qg_rep, sg, zg}, {qu_rep, su, zu}};
    cudaStream_t s = (cudaStream_t)stream;
    if (fused) return gemm_impl(A, sets, 2, sdt, Y, M, N, K, group, 0, s);

    const size_t need = w4a16_swiglu_workspace_bytes(M, N, K, group, 0);
    if (!ws || ws_bytes < need || !aligned(ws, 256)) return W4A16_ERR_WORKSPACE;
    Plan plan;
    if ((st = make_plan(M, N, K, group, 0, false, sdt == W4A16_SCALE_F32, &plan)) != W4A16_OK) return st;
    uint16_t *Gb = reinterpret_cast<uint16_t *>(ws);
    uint16_t *Ub = reinterpret_cast<uint16_t *>(reinterpret_cast<uint8_t *>(ws) +
                                                 align_up((size_t)M * N * 2, 256));
    if ((st = gemm_impl(A, &sets[0], 1, sdt, Gb, M, N, K, group, 0, s)) != W4A16_OK) return st;
    if ((st = gemm_impl(A, &sets[1], 1, sdt, Ub, M, N, K, group, 0, s)) != W4A16_OK) return st;
    return from_cuda(launch_silu_mul(reinterpret_cast<const __half *>(Gb),
                                     reinterpret_cast<const __half *>(Ub),
                                     reinterpret_cast<__half *>(Y), (size_t)M * N, s));
}

size_t w4a16_rmsnorm_workspace_bytes(int M, int N, int K, int group, int mode) {
    if (M <= 0 || N <= 0 || K <= 0 || mode < 0 || mode > 2) return 0;
    const size_t norm = align_up((size_t)M * K * 2, 256);
    return norm + (mode == 2 ? w4a16_swiglu_workspace_bytes(M, N, K, group, 0) : 0);
}

// Shared front half of the RMS-norm entry points: validates, stages the
// normalised activations at the start of ws and returns them.
static w4a16_status rmsnorm_prologue(const uint16_t *A, const uint16_t *gamma, float eps, int M, int N, int K,
                                     int group, int mode, void *ws, size_t ws_bytes, cudaStream_t s,
                                     uint16_t **An) {
    w4a16_status st = check_shape(M, N, K, group);
    if (st != W4A16_OK) return st;
    if (!A || !gamma || !aligned(A, 16) || !aligned(gamma, 16)) return W4A16_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || eps != eps) return W4A16_ERR_INVALID_ARG;
    if (!ws || !aligned(ws, 256) || ws_bytes < w4a16_rmsnorm_workspace_bytes(M, N, K, group, mode))
        return W4A16_ERR_WORKSPACE;
    *An = reinterpret_cast<uint16_t *>(ws);
    return W4A16_OK;
}

w4a16_status w4a16_gemm_rmsnorm(const uint16_t *A, const uint16_t *gamma, float eps, const uint8_t *q_rep,
                                const void *scales, w4a16_scale_dtype sdt, const uint8_t *zp, uint16_t *Y,
                                int M, int N, int K, int group, int split_k, void *ws, size_t ws_bytes,
                                void *stream) {
    cudaStream_t s = (cudaStream_t)stream;
    uint16_t *An = nullptr;
    w4a16_status st = rmsnorm_prologue(A, gamma, eps, M, N, K, group, 0, ws, ws_bytes, s, &An);
    if (st != W4A16_OK) return st;
    if (!Y || !aligned(Y, 16)) return W4A16_ERR_INVALID_ARG;
    if ((st = check_weights(q_rep, scales, sdt)) != W4A16_OK) return st;
    Plan plan;
    if ((st = make_plan(M, N, K, group, split_k, false, sdt == W4A16_SCALE_F32, &plan)) != W4A16_OK) return st;
    if (cudaError_t e = launch_rmsnorm(reinterpret_cast<const __half *>(A), reinterpret_cast<const __half *>(gamma),
                                       reinterpret_cast<__half *>(An), M, K, eps, g_launch_overlap != 0, s))
        return from_cuda(e);
    const WeightSet w{q_rep, scales, zp};
    return gemm_impl(An, &w, 1, sdt, Y, M, N, K, group, split_k, s);
}

w4a16_status w4a16_gemm_swiglu_rmsnorm(const uint16_t *A, const uint16_t *gamma, float eps,
                                       const uint8_t *qg_rep, const void *sg, const uint8_t *zg,
                                       const uint8_t *qu_rep, const void *su, const uint8_t *zu,
                                       w4a16_scale_dtype sdt, uint16_t *Y, int M, int N, int K, int group,
                                       int fused, void *ws, size_t ws_bytes, void *stream) {
    cudaStream_t s = (cudaStream_t)stream;
    uint16_t *An = nullptr;
    const int mode = fused ? 1 : 2;
    w4a16_status st = rmsnorm_prologue(A, gamma, eps, M, N, K, group, mode, ws, ws_bytes, s, &An);
    if (st != W4A16_OK) return st;
    if (!Y || !aligned(Y, 16)) return W4A16_ERR_INVALID_ARG;
    if ((st = check_weights(qg_rep, sg, sdt)) != W4A16_OK) return st;
    if ((st = check_weights(qu_rep, su, sdt)) != W4A16_OK) return st;
    Plan plan;
    if ((st = make_plan(M, N, K, group, 0, fused != 0, sdt == W4A16_SCALE_F32, &plan)) != W4A16_OK) return st;
    if (cudaError_t e = launch_rmsnorm(reinterpret_cast<const __half *>(A), reinterpret_cast<const __half *>(gamma),
                                       reinterpret_cast<__half *>(An), M, K, eps, g_launch_overlap != 0, s))
        return from_cuda(e);
    const size_t norm = align_up((size_t)M * K * 2, 256);
    void *rest = reinterpret_cast<uint8_t *>(ws) + norm;
    return w4a16_gemm_swiglu(An, qg_rep, sg, zg, qu_rep, su, zu, sdt, Y, M, N, K, group, fused, fused ? nullptr : rest,
                             fused ? 0 : ws_bytes - norm, stream);
}

w4a16_status w4a16_set_tuning(int smallm_max) {
    if (smallm_max < -1 || smallm_max > kSmallMMaxM) return W4A16_ERR_INVALID_ARG;
    g_smallm_max = smallm_max == 0 ? kSmallMMaxM : (smallm_max < 0 ? 0 : smallm_max);
    return W4A16_OK;
}

w4a16_status w4a16_set_launch_overlap(int enable) {
    if (enable != 0 && enable != 1) return W4A16_ERR_INVALID_ARG;
    g_launch_overlap = enable;
    return W4A16_OK;
}

w4a16_status w4a16_set_wait_limit_ns(unsigned long long limit_ns) {
    g_wait_ns = limit_ns;
    return W4A16_OK;
}

w4a16_status w4a16_device_error(void *stream) {
    unsigned int v = 0;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemcpyFromSymbolAsync(&v, g_device_error, sizeof(v), 0, cudaMemcpyDeviceToHost, s) !=
        cudaSuccess)
        return W4A16_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return W4A16_ERR_CUDA;
    if (v != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                    s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return W4A16_ERR_CUDA;
        return (w4a16_status)v;
    }
    return W4A16_OK;
}

}  // extern "C"
