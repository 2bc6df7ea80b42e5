// Internal declarations shared by the CUDA translation units of libw4a16.so.
// Not installed; the public interface is include/w4a16.h.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/w4a16.h"

namespace w4a16 {

// Repacked layout geometry (see w4a16_repack in include/w4a16.h).
constexpr int kTileRows = 128;   // rows per row tile
constexpr int kSubRows = 16;     // rows per sub-tile (one warp's MMA row block)
constexpr int kKBlock = 64;      // k per k-block
constexpr int kSubBytes = 512;   // bytes of one 16-row x 64-k sub-tile

// Byte offset of piece (16-row sub-tile S, k-block b): every sub-tile is one
// contiguous run of K/64 pieces of 512 bytes.
__host__ __device__ inline size_t piece_offset(int S, int b, int K) {
    return ((size_t)S * (size_t)(K / kKBlock) + (size_t)b) * (size_t)kSubBytes;
}

// ---------------------------------------------------------------------------
// Launch parameters
// ---------------------------------------------------------------------------
struct WeightSet {
    const uint8_t *q_rep;   // repacked int4 weights
    const void *scales;     // [N][G] fp16 or fp32
    const uint8_t *zp;      // [N][ceil(G/2)] or nullptr
};

struct SmallMParams {
    const __half *A;        // [M][K]
    WeightSet w[2];         // gate/up (w[1] only for SwiGLU)
    __half *Y;              // [M][N]
    int M, N, K, G;
    int scale_f32;
    int split;              // CTAs per row tile along K (cluster size; x2 for SwiGLU)
    int kc_blocks;          // k-blocks per staged activation chunk
    int overlap;            // launched as a programmatic dependent (weights read before the wait)
    unsigned int *err;      // device error word for bounded waits
    unsigned long long wait_ns;  // limit of each bounded wait
};

struct TcParams {
    const __half *A;
    WeightSet w[2];
    __half *Y;
    int M, N, K, G;
    int scale_f32;
    unsigned int *err;      // device error word for bounded waits
    unsigned long long wait_ns;  // limit of each bounded wait
};

// ---------------------------------------------------------------------------
// Tensor maps (TMA descriptors), encoded once per buffer and shape and cached.
// ---------------------------------------------------------------------------
struct TmapDesc {
    const void *ptr;
    int dtype;               // CUtensorMapDataType
    int rank;                // 2 or 3
    uint64_t dims[3];        // elements, innermost first
    uint64_t strides[2];     // bytes of dimensions 1 and 2
    uint32_t box[3];
    int swizzle128;          // 128-byte swizzle (else none)
};
bool encode_tmap(CUtensorMap *out, const TmapDesc &d);
// Repacked weights as (512-byte piece, k-block, sub-tile): a box of
// `kblocks_box` consecutive k-blocks of `subtiles_box` consecutive sub-tiles.
bool tmap_weights(CUtensorMap *out, const uint8_t *q_rep, int N, int K, int kblocks_box, int subtiles_box);
// Activations [M][K] fp16: boxes of 64 k x rows_box tokens, 128-byte swizzle,
// tokens past M read as zero.
bool tmap_activations(CUtensorMap *out, const __half *A, int M, int K, int rows_box);
// The same activations as (64 k, token, k-block): one box brings `kblocks_box`
// consecutive k-blocks of rows_box tokens, laid out k-block after k-block.
bool tmap_activations_kblocks(CUtensorMap *out, const __half *A, int M, int K, int rows_box, int kblocks_box);

// Number of SMs of the current device (cached per device, thread-safe).
int sm_count();

// Raise `func`'s dynamic shared-memory limit to `bytes` once per device
// (thread-safe; later calls for the same kernel and device do nothing).
cudaError_t ensure_max_dyn_smem(const void *func, int bytes);

// Host-side launchers (return cudaError_t of the launch).
cudaError_t launch_repack(const uint8_t *q, uint8_t *q_rep, int N, int K, cudaStream_t s);

struct SmallMPlan {
    int split;      // CTAs per row tile along K (cluster size, 1..8)
    int kc;         // k-blocks per staged activation chunk
    int smem;       // dynamic shared memory per CTA (bytes)
    int per_sm;     // resident CTAs per SM at that shared-memory size
};
SmallMPlan smallm_plan(int M, int N, int K, int group, bool swiglu, int split_k, int sm_count);
cudaError_t launch_smallm(const SmallMParams &p, int group, bool swiglu, cudaStream_t s);
cudaError_t launch_tc(const TcParams &p, int group, bool swiglu, cudaStream_t s);
int tc_tile_tokens(int M, bool swiglu);
// Launch shape of the tensor-core kernel: CTAs, threads, dynamic shared memory, ring stages.
void tc_launch_shape(int M, int N, bool swiglu, int *ctas, int *threads, int *smem, int *stages);
// Threads per CTA of the small-M tile kernel.
int smallm_threads(int M, bool swiglu);
cudaError_t launch_rmsnorm(const __half *A, const __half *gamma, __half *An, int M, int K, float eps, bool overlap,
                           cudaStream_t s);
cudaError_t launch_silu_mul(const __half *G, const __half *U, __half *Y, size_t n,
                            cudaStream_t s);

constexpr int kSmallMMaxM = 64;      // 8 token tiles of 8

}  // namespace w4a16
