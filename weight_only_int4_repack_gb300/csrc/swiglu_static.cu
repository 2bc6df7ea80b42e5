// Unfused SwiGLU for callers that cannot allocate device memory.
//
// The unfused chain (gate GEMM -> fp16 G, up GEMM -> fp16 U, silu_mul -> Y)
// needs 4*M*N bytes of scratch for G and U. Some callers have no way to provide
// it: code running inside another framework's memory pool that may not call
// cudaMalloc, hot paths where a device allocation (which can synchronise the
// device) is not acceptable, or plug-ins handed only input and output buffers.
// This entry point keeps that scratch in a fixed array compiled into the
// library, so a call allocates nothing; inputs and outputs still come from the
// caller. The array exists once per GPU that loads the library and stays
// allocated until the process exits.
#include <mutex>

#include "w4a16_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = (size_t)8 << 20;  // 8 MiB: 4*M*N <= this

// Shared by every call on a device; the last call's G and U stay in it.
static __device__ __align__(256) unsigned char g_swiglu_scratch[kStaticScratchBytes];

// Device address of the array on the current device. In host code the symbol
// names a host-side shadow, not device memory, so the address must come from
// cudaGetSymbolAddress, once per device, with that device current.
unsigned char *scratch_address(w4a16_status *st) {
    static std::mutex mu;
    static unsigned char *cached[64] = {nullptr};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *st = W4A16_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_swiglu_scratch) != cudaSuccess || ptr == nullptr) {
            *st = W4A16_ERR_CUDA;
            return nullptr;
        }
        cached[dev] = static_cast<unsigned char *>(ptr);
    }
    *st = W4A16_OK;
    return cached[dev];
}

}  // namespace

extern "C" {

size_t w4a16_swiglu_static_scratch_bytes(void) { return kStaticScratchBytes; }

w4a16_status w4a16_gemm_swiglu_unfused_static(const uint16_t *A,
                                              const uint8_t *qg_rep, const void *sg, const uint8_t *zg,
                                              const uint8_t *qu_rep, const void *su, const uint8_t *zu,
                                              w4a16_scale_dtype sdt, uint16_t *Y,
                                              int M, int N, int K, int group, void *stream) {
    if (M <= 0 || N <= 0 || K <= 0) return W4A16_ERR_INVALID_ARG;
    const size_t need = w4a16_swiglu_workspace_bytes(M, N, K, group, 0);
    if (need > kStaticScratchBytes) return W4A16_ERR_WORKSPACE;  // 4*M*N exceeds the fixed array
    w4a16_status st = W4A16_OK;
    unsigned char *scratch = scratch_address(&st);
    if (!scratch) return st;
    // G and U are written in full before they are read: nothing needs clearing.
    return w4a16_gemm_swiglu(A, qg_rep, sg, zg, qu_rep, su, zu, sdt, Y, M, N, K, group, /*fused=*/0,
                             scratch, kStaticScratchBytes, stream);
}

}  // extern "C"
