// Small-M W4A16 GEMM (decode / verify shapes, M <= 64): a weight-streaming kernel.
//
// At small M the GEMM is bound by reading the int4 weights once from HBM. The
// MatMulNBits Marlin pull request (github.com/justinchuby/onnx-genai pull 960,
// "P2 -- widen the win: split-K" and "Small-M split-K retune") found small M
// occupancy-bound and split the K range over more CTAs, reducing fp32 partials
// in a fixed order. This kernel keeps those two ideas and re-designs the rest
// for sm_103a:
//   * one CTA = one 128-row tile (8 warps x 16-row sub-tiles) x one K range;
//     every lane streams its sub-tile with 128-bit coalesced loads (512 contiguous
//     bytes per warp per 64-k block), kSmallMPrefetch blocks in flight per warp;
//   * the repacked words are already mma.sync.m16n8k16 A fragments: one and/or
//     per half2 turns two nibbles into fp16 (1024 + q), one sub.f16x2 removes
//     (1024 + zp) exactly, tokens are the n=8 operand (fp32 accumulation);
//   * the group scale is applied to each group's fp32 partial sum (the pull
//     request's "per-group scale AFTER the tensor-core accumulate");
//   * the K split is a thread-block cluster: partial tiles are summed through
//     distributed shared memory in rank order (deterministic, no global scratch,
//     one launch).
// CUDA-core FMA would need M FMAs per weight; at M = 8 that is about 0.57 G FMA
// for K=5120, N=13824, more than the FP32 pipes finish in the HBM time of the
// weight stream, so the contraction runs on the tensor cores.
#include "w4a16_internal.h"

namespace w4a16 {
namespace {

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t sub_f16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// D = A(16x16, row) * B(16x8, col) + C, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1, const float (&c)[4]) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
          "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ float ld_dsmem_f32(const float *local, uint32_t rank) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(local);
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(s), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

__device__ __forceinline__ float silu_f32(float x) { return x / (1.0f + expf(-x)); }

// Shared-memory plan of one CTA (all offsets in bytes from the dynamic base).
struct SmemPlan {
    int a_stride;      // halves per staged activation row: kc*64 + 16
    int ng;            // group slots per staged chunk
    size_t a_bytes, meta_bytes_per_set, part_stride_floats;
};

__host__ __device__ inline SmemPlan make_plan(int MT, int group, int kc_blocks, int nsets) {
    SmemPlan p;
    p.a_stride = kc_blocks * kKBlock + 16;  // +32 bytes: conflict-free 8-byte fragment loads
    p.ng = (kc_blocks * kKBlock) / group + 1;
    p.a_bytes = (size_t)8 * MT * p.a_stride * 2;
    p.meta_bytes_per_set = (size_t)kTileRows * p.ng * 8;  // float scale + half2 (1024+zp)
    p.part_stride_floats = kTileRows + 4;
    (void)nsets;
    return p;
}

template <int GROUP, int MT, bool SWIGLU>
__global__ void __launch_bounds__(kSmallMThreads, (MT * (SWIGLU ? 2 : 1) <= 2) ? 2 : 1)
    smallm_kernel(const SmallMParams p) {
    constexpr int NS = SWIGLU ? 2 : 1;
    constexpr int PF = SWIGLU ? kSmallMPrefetch / 2 : kSmallMPrefetch;
    constexpr int FL = GROUP < kKBlock ? GROUP : kKBlock;  // k per scale flush
    constexpr int SPF = FL / 16;                             // k16 steps per flush

    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;

    const int n0 = blockIdx.x * kTileRows;
    const int R = min(kTileRows, p.N - n0);
    const int nsub = R / kSubRows;
    const int s = warp;                      // this warp's sub-tile
    const bool active = s < nsub;

    const int S = p.split;
    const int rank = (S > 1) ? (int)cluster_rank() : 0;
    const int nb = p.K / kKBlock;
    const int b_begin = (int)((long long)nb * rank / S);
    const int b_end = (int)((long long)nb * (rank + 1) / S);
    const int kc = p.kc_blocks;

    const SmemPlan plan = make_plan(MT, GROUP, kc, NS);
    __half *sA = reinterpret_cast<__half *>(smem);
    float *sSc = reinterpret_cast<float *>(smem + plan.a_bytes);
    uint32_t *sZp = reinterpret_cast<uint32_t *>(smem + plan.a_bytes) + (size_t)kTileRows * plan.ng;
    const size_t meta_set_words = plan.meta_bytes_per_set / 4;

    // Zero the activation rows beyond M once (they stay zero for every chunk).
    for (int m = p.M; m < 8 * MT; ++m)
        for (int i = tid; i < plan.a_stride; i += kSmallMThreads) sA[(size_t)m * plan.a_stride + i] = __float2half(0.f);

    // Weight stream pointers: chunk stride R*32 bytes per k-block.
    const size_t tile_base = (size_t)n0 * (size_t)(p.K / 2) + (size_t)s * kSubBytes + (size_t)lane * 16;
    const size_t bstride = (size_t)R * 32;
    const uint8_t *wptr[NS];
#pragma unroll
    for (int w = 0; w < NS; ++w) wptr[w] = p.w[w].q_rep + tile_base;

    uint4 buf[NS][PF];
#pragma unroll
    for (int i = 0; i < PF; ++i)
#pragma unroll
        for (int w = 0; w < NS; ++w)
            if (active && b_begin + i < b_end) buf[w][i] = ldg_stream(wptr[w] + (size_t)(b_begin + i) * bstride);

    float acc[NS][MT][4];
#pragma unroll
    for (int w = 0; w < NS; ++w)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[w][mt][i] = 0.f;

    const int rg = s * kSubRows + g;  // row (in tile) of fragment half 0; half 1 is rg + 8
    const int zpstride = (p.G + 1) / 2;

    for (int c0 = b_begin; c0 < b_end; c0 += kc) {
        const int c1 = min(c0 + kc, b_end);
        const int grp0 = (c0 * kKBlock) / GROUP;
        const int ng = ((c1 * kKBlock - 1) / GROUP) - grp0 + 1;
        __syncthreads();  // previous chunk fully consumed
        // Stage activations [M][c0*64, c1*64) with 16-byte async copies.
        {
            const int kl = (c1 - c0) * kKBlock;
            const int per_row = kl / 8;
            for (int i = tid; i < p.M * per_row; i += kSmallMThreads) {
                const int m = i / per_row, q = i % per_row;
                cp_async16(sA + (size_t)m * plan.a_stride + q * 8,
                           p.A + (size_t)m * p.K + (size_t)c0 * kKBlock + q * 8);
            }
        }
        // Stage scales (as float) and zero points (as half2 of 1024 + zp) of the chunk's groups.
#pragma unroll
        for (int w = 0; w < NS; ++w) {
            float *sc = sSc + w * meta_set_words;
            uint32_t *zz = sZp + w * meta_set_words;
            const uint8_t *zpg = p.w[w].zp;
            for (int i = tid; i < R * ng; i += kSmallMThreads) {
                const int row = i / ng, gi = i % ng;
                const int n = n0 + row, grp = grp0 + gi;
                float sv = 0.f;
                uint32_t zv = 8;
                if (grp < p.G) {
                    const size_t si = (size_t)n * p.G + grp;
                    sv = p.scale_f32 ? __ldg(reinterpret_cast<const float *>(p.w[w].scales) + si)
                                     : __half2float(__ldg(reinterpret_cast<const __half *>(p.w[w].scales) + si));
                    if (zpg) {
                        const uint8_t zb = __ldg(zpg + (size_t)n * zpstride + (grp >> 1));
                        zv = (grp & 1) ? (zb >> 4) : (zb & 0xF);
                    }
                }
                const uint32_t h = 0x6400u + zv;  // fp16 bits of 1024 + zp
                sc[row * plan.ng + gi] = sv;
                zz[row * plan.ng + gi] = h | (h << 16);
            }
        }
        cp_async_wait_all();
        __syncthreads();

        for (int bb = c0; bb < c1; bb += PF) {
#pragma unroll
            for (int i = 0; i < PF; ++i) {
                const int b = bb + i;
                if (b < c1 && active) {
                    uint4 wv[NS];
#pragma unroll
                    for (int w = 0; w < NS; ++w) {
                        wv[w] = buf[w][i];
                        if (b + PF < b_end) buf[w][i] = ldg_stream(wptr[w] + (size_t)(b + PF) * bstride);
                    }
                    const int kl = (b - c0) * kKBlock;
                    float accg[NS][MT][4];
                    uint32_t zz0[NS], zz1[NS];
                    float sc0[NS], sc1[NS];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (j % SPF == 0) {
                            const int gi = ((b * kKBlock + 16 * j) / GROUP) - grp0;
#pragma unroll
                            for (int w = 0; w < NS; ++w) {
                                const float *sc = sSc + w * meta_set_words;
                                const uint32_t *zz = sZp + w * meta_set_words;
                                zz0[w] = zz[rg * plan.ng + gi];
                                zz1[w] = zz[(rg + 8) * plan.ng + gi];
                                sc0[w] = sc[rg * plan.ng + gi];
                                sc1[w] = sc[(rg + 8) * plan.ng + gi];
                            }
                        }
                        // Activation fragment for each token tile: k = 16j + 4t .. +3.
                        uint32_t bfr[MT][2];
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            const uint2 v = *reinterpret_cast<const uint2 *>(
                                sA + (size_t)(8 * mt + g) * plan.a_stride + kl + 16 * j + 4 * t);
                            bfr[mt][0] = v.x;
                            bfr[mt][1] = v.y;
                        }
#pragma unroll
                        for (int w = 0; w < NS; ++w) {
                            const uint32_t word = (&wv[w].x)[j];
                            uint32_t a[4];
                            a[0] = sub_f16x2((word & 0x000F000Fu) | 0x64006400u, zz0[w]);
                            a[1] = sub_f16x2(((word >> 4) & 0x000F000Fu) | 0x64006400u, zz1[w]);
                            a[2] = sub_f16x2(((word >> 8) & 0x000F000Fu) | 0x64006400u, zz0[w]);
                            a[3] = sub_f16x2(((word >> 12) & 0x000F000Fu) | 0x64006400u, zz1[w]);
#pragma unroll
                            for (int mt = 0; mt < MT; ++mt) {
                                if (j % SPF == 0) {
                                    const float z4[4] = {0.f, 0.f, 0.f, 0.f};
                                    mma_16816(accg[w][mt], a, bfr[mt][0], bfr[mt][1], z4);
                                } else {
                                    mma_16816(accg[w][mt], a, bfr[mt][0], bfr[mt][1], accg[w][mt]);
                                }
                            }
                            if (j % SPF == SPF - 1) {
#pragma unroll
                                for (int mt = 0; mt < MT; ++mt) {
                                    acc[w][mt][0] = fmaf(sc0[w], accg[w][mt][0], acc[w][mt][0]);
                                    acc[w][mt][1] = fmaf(sc0[w], accg[w][mt][1], acc[w][mt][1]);
                                    acc[w][mt][2] = fmaf(sc1[w], accg[w][mt][2], acc[w][mt][2]);
                                    acc[w][mt][3] = fmaf(sc1[w], accg[w][mt][3], acc[w][mt][3]);
                                }
                            }
                        }
                    }
                }
            }
        }
    }

    // Partial tile -> shared memory as [set][token][row] (row stride 132 floats).
    __syncthreads();
    float *P = reinterpret_cast<float *>(smem);
    const size_t set_floats = (size_t)8 * MT * plan.part_stride_floats;
    if (active) {
#pragma unroll
        for (int w = 0; w < NS; ++w)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                float *Pw = P + w * set_floats;
                const int m0 = 8 * mt + 2 * t;
                Pw[(size_t)m0 * plan.part_stride_floats + rg] = acc[w][mt][0];
                Pw[(size_t)(m0 + 1) * plan.part_stride_floats + rg] = acc[w][mt][1];
                Pw[(size_t)m0 * plan.part_stride_floats + rg + 8] = acc[w][mt][2];
                Pw[(size_t)(m0 + 1) * plan.part_stride_floats + rg + 8] = acc[w][mt][3];
            }
    }
    if (S > 1) cluster_sync(); else __syncthreads();

    // Rank r finalises rows [r*R/S, (r+1)*R/S): sum partials of ranks 0..S-1 in order.
    const int lo = (int)((long long)R * rank / S), hi = (int)((long long)R * (rank + 1) / S);
    const int nr = hi - lo;
    for (int i = tid; i < p.M * nr; i += kSmallMThreads) {
        const int m = i / nr, row = lo + i % nr;
        float v[NS];
#pragma unroll
        for (int w = 0; w < NS; ++w) {
            const float *src = P + w * set_floats + (size_t)m * plan.part_stride_floats + row;
            if (S > 1) {
                float sum = ld_dsmem_f32(src, 0);
                for (int q = 1; q < S; ++q) sum += ld_dsmem_f32(src, q);
                v[w] = sum;
            } else {
                v[w] = *src;
            }
        }
        float y = v[0];
        if constexpr (SWIGLU) y = silu_f32(v[0]) * v[1];
        p.Y[(size_t)m * p.N + n0 + row] = __float2half_rn(y);
    }
    if (S > 1) cluster_sync();  // keep shared memory alive until every peer has read it
}

template <int GROUP, int MT, bool SWIGLU>
cudaError_t launch_one(const SmallMParams &p, cudaStream_t s) {
    const size_t smem = smallm_smem_bytes(p.M, GROUP, SWIGLU, p.kc_blocks);
    auto kern = smallm_kernel<GROUP, MT, SWIGLU>;
    static size_t configured = 0;  // per instantiation; attribute is per device-agnostic function
    if (smem > configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.N + kTileRows - 1) / kTileRows), (unsigned)p.split, 1);
    cfg.blockDim = dim3(kSmallMThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)p.split;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.split > 1 ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int GROUP, bool SWIGLU>
cudaError_t launch_mt(const SmallMParams &p, cudaStream_t s) {
    const int mt = (p.M + 7) / 8;
    if (mt <= 1) return launch_one<GROUP, 1, SWIGLU>(p, s);
    if (mt <= 2) return launch_one<GROUP, 2, SWIGLU>(p, s);
    if (mt <= 4) return launch_one<GROUP, 4, SWIGLU>(p, s);
    return launch_one<GROUP, 8, SWIGLU>(p, s);
}

template <bool SWIGLU>
cudaError_t launch_group(const SmallMParams &p, int group, cudaStream_t s) {
    switch (group) {
        case 16: return launch_mt<16, SWIGLU>(p, s);
        case 32: return launch_mt<32, SWIGLU>(p, s);
        case 64: return launch_mt<64, SWIGLU>(p, s);
        default: return launch_mt<128, SWIGLU>(p, s);
    }
}

int mt_of(int M) {
    const int mt = (M + 7) / 8;
    return mt <= 1 ? 1 : mt <= 2 ? 2 : mt <= 4 ? 4 : 8;
}

}  // namespace

size_t smallm_smem_bytes(int M, int group, bool swiglu, int kc_blocks) {
    const int MT = mt_of(M);
    const int ns = swiglu ? 2 : 1;
    const SmemPlan pl = make_plan(MT, group, kc_blocks, ns);
    const size_t stage = pl.a_bytes + ns * pl.meta_bytes_per_set;
    const size_t part = (size_t)ns * 8 * MT * pl.part_stride_floats * 4;
    return stage > part ? stage : part;
}

// Largest chunk (in k-blocks, a multiple of the prefetch depth) that keeps one
// CTA's shared memory within the budget for two resident CTAs per SM.
int smallm_max_kc(int M, int group, bool swiglu) {
    const size_t budget = 100 * 1024;
    int kc = kSmallMPrefetch;
    while (smallm_smem_bytes(M, group, swiglu, kc + kSmallMPrefetch) <= budget && kc < 1024)
        kc += kSmallMPrefetch;
    return kc;
}

cudaError_t launch_smallm(const SmallMParams &p, int group, bool swiglu, cudaStream_t s) {
    return swiglu ? launch_group<true>(p, group, s) : launch_group<false>(p, group, s);
}

}  // namespace w4a16
