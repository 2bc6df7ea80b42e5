// Device repack of nibble-packed int4 weights into the fragment-interleaved layout
// (16-row sub-tiles, each one contiguous run of 512-byte pieces along K).
//
// The MatMulNBits Marlin pull request (github.com/justinchuby/onnx-genai pull 960,
// "What's landed") repacks the ONNX nibble format once, on the device, into a
// bijective interleaved order so that warps load contiguous bytes; its device
// repack is byte-identical to a host reference. This is the same idea for this
// library's own layout (stated in include/w4a16.h). Integer work, HBM-bound:
// every thread produces one 16-byte lane slot (two rows x 16 k of four k16
// steps) and writes it with one coalesced 128-bit store.
#include "w4a16_internal.h"

namespace w4a16 {

__global__ void __launch_bounds__(256) repack_kernel(const uint8_t *__restrict__ q,
                                                     uint4 *__restrict__ out, int N, int K,
                                                     long long n_chunks) {
    long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= n_chunks) return;
    // 16-byte chunk c is lane slot c % 32 of piece c / 32 = (sub-tile S, k-block b).
    const long long piece = c >> 5;
    const int kblocks = K / kKBlock;
    const int S = (int)(piece / kblocks);
    const int b = (int)(piece % kblocks);
    const int slot = (int)(c & 31);
    // Slot 4g + (t + g/2) % 4 holds the fragment owned by (g, t).
    const int g = slot >> 2, t = ((slot & 3) - (g >> 1)) & 3;
    const size_t row_bytes = (size_t)(K / 2);
    const uint8_t *r0 = q + (size_t)(S * kSubRows + g) * row_bytes;
    const uint8_t *r1 = r0 + 8 * row_bytes;
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int kb = (b * kKBlock + 16 * j + 4 * t) / 2;   // byte of k = ... + 4t (even)
        const uint32_t x0 = *reinterpret_cast<const uint16_t *>(r0 + kb);  // e0..e3 of row g
        const uint32_t x1 = *reinterpret_cast<const uint16_t *>(r1 + kb);  // e0..e3 of row g+8
        // Nibble p of the word holds element e of row half h at p = 4(e%2) + 2(e/2) + h.
        uint32_t word = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int p = 4 * (e & 1) + 2 * (e >> 1);
            word |= ((x0 >> (4 * e)) & 0xFu) << (4 * p);
            word |= ((x1 >> (4 * e)) & 0xFu) << (4 * (p + 1));
        }
        w[j] = word;
    }
    out[c] = make_uint4(w[0], w[1], w[2], w[3]);
}

cudaError_t launch_repack(const uint8_t *q, uint8_t *q_rep, int N, int K, cudaStream_t s) {
    const long long n_chunks = (long long)N * K / 32;
    const int threads = 256;
    const long long blocks = (n_chunks + threads - 1) / threads;
    repack_kernel<<<(unsigned)blocks, threads, 0, s>>>(q, reinterpret_cast<uint4 *>(q_rep), N, K,
                                                        n_chunks);
    return cudaGetLastError();
}

}  // namespace w4a16
