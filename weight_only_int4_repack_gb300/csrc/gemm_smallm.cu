// Small-M W4A16 GEMM (decode / verify shapes, M <= 64): a weight-streaming kernel.
//
// At small M the GEMM is bound by reading the int4 weights once from HBM. The
// MatMulNBits Marlin pull request (github.com/justinchuby/onnx-genai pull 960,
// "P2 -- widen the win: split-K" and "Small-M split-K retune") found small M
// occupancy-bound and split the K range over more CTAs, reducing fp32 partials
// in a fixed order. This kernel keeps those two ideas and re-designs the rest
// for sm_103a:
//   * one CTA = one 128-row tile (8 consumer warps, one 16-row sub-tile each) x
//     one K range, plus a producer warp. The producer streams each (tile, 64-k
//     block) chunk -- 4 KB contiguous in the repacked layout -- into a 48 KB
//     shared-memory ring with cp.async.bulk (the TMA engine), so tens of KB per
//     CTA are in flight without costing registers;
//   * each consumer lane reads one 16-byte slot (a 128-bit, conflict-free shared
//     load); its four words are already mma.sync.m16n8k16 A fragments: one
//     and/or per half2 turns two nibbles into fp16 (1024 + q), one sub.f16x2
//     removes (1024 + zp) exactly, and the tokens are the n=8 operand;
//   * fp32 accumulation; the group scale is applied to each group's fp32 partial
//     sum (the pull request's "per-group scale AFTER the tensor-core accumulate");
//   * the K split is a thread-block cluster: partial tiles are summed through
//     distributed shared memory in rank order (deterministic, no global scratch,
//     one launch).
// CUDA-core FMA would need M FMAs per weight; at M = 8 that is about 0.57 G FMA
// for K=5120, N=13824, more than the FP32 pipes finish in the HBM time of the
// weight stream, so the contraction runs on the tensor cores.
#include "ptx.cuh"
#include "w4a16_internal.h"

namespace w4a16 {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kRingBytes = 48 * 1024;
constexpr int kChunkMax = kTileRows * 32;  // bytes of one (tile, k-block) chunk
constexpr int kPartStride = kTileRows + 4;  // floats per partial row (bank spread)

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

__device__ __forceinline__ float silu_f32(float x) { return x / (1.0f + expf(-x)); }

// Shared-memory plan of one CTA (byte offsets from the dynamic base).
struct SmemPlan {
    int stages, a_stride, ng;
    size_t a_off, meta_off, meta_set_bytes, bar_off, total;
};

__host__ __device__ inline SmemPlan make_plan(int MT, int group, int kc, int ns) {
    SmemPlan p;
    p.stages = kRingBytes / (ns * kChunkMax);
    p.a_off = (size_t)p.stages * ns * kChunkMax;
    p.a_stride = kc * kKBlock + 16;  // +32 bytes per row: conflict-free 8-byte fragment loads
    p.ng = (kc * kKBlock) / group + 1;
    p.meta_off = p.a_off + (size_t)8 * MT * p.a_stride * 2;
    p.meta_set_bytes = (size_t)kTileRows * p.ng * 8;  // float scale + half2 (1024 + zp)
    const size_t main_end = p.meta_off + ns * p.meta_set_bytes;
    const size_t part_end = (size_t)ns * 8 * MT * kPartStride * 4;  // aliases the ring after use
    const size_t end = main_end > part_end ? main_end : part_end;
    p.bar_off = (end + 15) / 16 * 16;
    p.total = p.bar_off + (size_t)(2 * p.stages + 2) * 8;
    return p;
}

template <int MT, bool SWIGLU>
struct MinBlocks {
    static constexpr int value = (MT * (SWIGLU ? 2 : 1) <= 4) ? 2 : 1;
};

template <int GROUP, int MT, bool SWIGLU>
__global__ void __launch_bounds__(kSmallMThreads, (MinBlocks<MT, SWIGLU>::value))
    smallm_kernel(const SmallMParams p) {
    constexpr int NS = SWIGLU ? 2 : 1;
    constexpr int FL = GROUP < kKBlock ? GROUP : kKBlock;  // k per scale flush
    constexpr int SPF = FL / 16;                             // k16 steps per flush

    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    const int n0 = blockIdx.x * kTileRows;
    const int R = min(kTileRows, p.N - n0);
    const int nsub = R / kSubRows;
    const int S = p.split;
    const int rank = (S > 1) ? (int)ptx::cluster_rank() : 0;
    const int nb = p.K / kKBlock;
    const int b_begin = (int)((long long)nb * rank / S);
    const int b_end = (int)((long long)nb * (rank + 1) / S);
    const int nblk = b_end - b_begin;
    const int kc = p.kc_blocks;
    const SmemPlan plan = make_plan(MT, GROUP, kc, NS);
    const int stages = plan.stages;

    uint64_t *full = reinterpret_cast<uint64_t *>(smem + plan.bar_off);
    uint64_t *empty = full + stages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + stages);
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        ptx::mbar_init_fence();
    }
    __syncthreads();

    const uint32_t chunk_bytes = (uint32_t)R * 32u;
    float *P = reinterpret_cast<float *>(smem);  // partial tile, valid after the main loop
    const size_t set_floats = (size_t)8 * MT * kPartStride;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int it = 0;
            for (; it < nblk; ++it) {
                const int s = it % stages;
                const uint32_t ph = (uint32_t)(it / stages) & 1u;
                if (!ptx::mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.err)) break;
                ptx::mbar_arrive_expect_tx(&full[s], NS * chunk_bytes);
                const size_t off = chunk_offset(n0, p.N, p.K, b_begin + it);
#pragma unroll
                for (int w = 0; w < NS; ++w)
                    ptx::bulk_g2s(smem + (size_t)(s * NS + w) * kChunkMax, p.w[w].q_rep + off, chunk_bytes,
                                  &full[s]);
            }
            if (*abort_flag) {
                // Let the copies already issued land before the CTA can exit.
                volatile int no_abort = 0;
                for (int s = 0; s < stages && s < it; ++s) {
                    const int last = s + ((it - 1 - s) / stages) * stages;
                    ptx::mbar_wait(&full[s], (uint32_t)(last / stages) & 1u, &no_abort, nullptr,
                                   200000000ull);
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ consumers
        const int g = lane >> 2, t = lane & 3;
        const int slot = 4 * g + ((t + (g >> 1)) & 3);  // lane slot of fragment (g, t)
        const int cw = warp;                             // sub-tile of this warp
        const bool active = cw < nsub;
        const int rg = cw * kSubRows + g;                // tile row of fragment half 0
        const int zpstride = (p.G + 1) / 2;

        __half *sA = reinterpret_cast<__half *>(smem + plan.a_off);
        float *sSc = reinterpret_cast<float *>(smem + plan.meta_off);
        const size_t meta_words = plan.meta_set_bytes / 4;  // per set: ng*128 floats + ng*128 words

        for (int m = p.M; m < 8 * MT; ++m)
            for (int i = tid; i < plan.a_stride; i += kConsumers)
                sA[(size_t)m * plan.a_stride + i] = __float2half(0.f);

        float acc[NS][MT][4];
#pragma unroll
        for (int w = 0; w < NS; ++w)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[w][mt][i] = 0.f;

        bool aborted = false;
        for (int c0 = b_begin; c0 < b_end; c0 += kc) {
            const int c1 = min(c0 + kc, b_end);
            const int grp0 = (c0 * kKBlock) / GROUP;
            const int ng = ((c1 * kKBlock - 1) / GROUP) - grp0 + 1;
            ptx::named_bar_sync(1, kConsumers);  // previous chunk consumed
            {   // activations [M][c0*64, c1*64): 16-byte async copies
                const int per_row = (c1 - c0) * kKBlock / 8;
                for (int i = tid; i < p.M * per_row; i += kConsumers) {
                    const int m = i / per_row, q = i % per_row;
                    ptx::cp_async16(sA + (size_t)m * plan.a_stride + q * 8,
                                    p.A + (size_t)m * p.K + (size_t)c0 * kKBlock + q * 8);
                }
            }
            // Scales (as float) and zero points (as half2 of 1024 + zp): all loads
            // of a batch are issued before any is used.
#pragma unroll
            for (int w = 0; w < NS; ++w) {
                float *sc = sSc + w * meta_words;
                uint32_t *zz = reinterpret_cast<uint32_t *>(sc) + (size_t)kTileRows * plan.ng;
                const uint8_t *zpg = p.w[w].zp;
                const int total = R * ng;
                for (int base = 0; base < total; base += kConsumers * 8) {
                    float sv[8];
                    uint32_t zb[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int i = base + tid + kConsumers * u;
                        sv[u] = 0.f;
                        zb[u] = 0x88u;
                        if (i < total) {
                            const int row = i / ng, gi = i % ng;
                            const int grp = grp0 + gi;
                            if (grp < p.G) {
                                const size_t si = (size_t)(n0 + row) * p.G + grp;
                                sv[u] = p.scale_f32
                                            ? __ldg(reinterpret_cast<const float *>(p.w[w].scales) + si)
                                            : __half2float(__ldg(reinterpret_cast<const __half *>(p.w[w].scales) + si));
                                if (zpg) zb[u] = __ldg(zpg + (size_t)(n0 + row) * zpstride + (grp >> 1));
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int i = base + tid + kConsumers * u;
                        if (i < total) {
                            const int row = i / ng, gi = i % ng;
                            const uint32_t zv = ((grp0 + gi) & 1) ? (zb[u] >> 4) : (zb[u] & 0xFu);
                            const uint32_t h = 0x6400u + zv;  // fp16 bits of 1024 + zp
                            sc[row * plan.ng + gi] = sv[u];
                            zz[row * plan.ng + gi] = h | (h << 16);
                        }
                    }
                }
            }
            ptx::cp_async_wait_all();
            ptx::named_bar_sync(1, kConsumers);

            for (int b = c0; b < c1; ++b) {
                const int it = b - b_begin;
                const int s = it % stages;
                const uint32_t ph = (uint32_t)(it / stages) & 1u;
                if (!aborted && !ptx::mbar_wait(&full[s], ph, abort_flag, p.err)) aborted = true;
                if (aborted) continue;
                uint4 wv[NS];
                if (active) {
#pragma unroll
                    for (int w = 0; w < NS; ++w)
                        wv[w] = *reinterpret_cast<const uint4 *>(smem + (size_t)(s * NS + w) * kChunkMax +
                                                                 cw * kSubBytes + slot * 16);
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&empty[s]);
                if (!active) continue;

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
                            const float *sc = sSc + w * meta_words;
                            const uint32_t *zz = reinterpret_cast<const uint32_t *>(sc) + (size_t)kTileRows * plan.ng;
                            zz0[w] = zz[rg * plan.ng + gi];
                            zz1[w] = zz[(rg + 8) * plan.ng + gi];
                            sc0[w] = sc[rg * plan.ng + gi];
                            sc1[w] = sc[(rg + 8) * plan.ng + gi];
                        }
                    }
                    // Activation fragment of each token tile: k = 16j + 4t .. +3.
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

        // Partial tile -> shared memory as [set][token][row]; it overlays the ring
        // and the staging area, which every consumer warp has finished with.
        ptx::named_bar_sync(1, kConsumers);
        if (active) {
#pragma unroll
            for (int w = 0; w < NS; ++w)
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    float *Pw = P + w * set_floats;
                    const int m0 = 8 * mt + 2 * t;
                    Pw[(size_t)m0 * kPartStride + rg] = acc[w][mt][0];
                    Pw[(size_t)(m0 + 1) * kPartStride + rg] = acc[w][mt][1];
                    Pw[(size_t)m0 * kPartStride + rg + 8] = acc[w][mt][2];
                    Pw[(size_t)(m0 + 1) * kPartStride + rg + 8] = acc[w][mt][3];
                }
        }
    }

    if (S > 1) ptx::cluster_sync(); else __syncthreads();

    // Rank r finalises rows [r*R/S, (r+1)*R/S): partials of ranks 0..S-1 summed in order.
    if (tid < kConsumers) {
        const int lo = (int)((long long)R * rank / S), hi = (int)((long long)R * (rank + 1) / S);
        const int nr = hi - lo;
        for (int i = tid; i < p.M * nr; i += kConsumers) {
            const int m = i / nr, row = lo + i % nr;
            float v[NS];
#pragma unroll
            for (int w = 0; w < NS; ++w) {
                const float *src = P + w * set_floats + (size_t)m * kPartStride + row;
                if (S > 1) {
                    float sum = ptx::ld_dsmem_f32(src, 0);
                    for (int q = 1; q < S; ++q) sum += ptx::ld_dsmem_f32(src, (uint32_t)q);
                    v[w] = sum;
                } else {
                    v[w] = *src;
                }
            }
            float y = v[0];
            if constexpr (SWIGLU) y = silu_f32(v[0]) * v[1];
            p.Y[(size_t)m * p.N + n0 + row] = __float2half_rn(y);
        }
    }
    if (S > 1) ptx::cluster_sync();  // keep shared memory alive until every peer has read it
}

template <int GROUP, int MT, bool SWIGLU>
cudaError_t launch_one(const SmallMParams &p, cudaStream_t s) {
    const size_t smem = make_plan(MT, GROUP, p.kc_blocks, SWIGLU ? 2 : 1).total;
    auto kern = smallm_kernel<GROUP, MT, SWIGLU>;
    static size_t configured = 0;
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
    return make_plan(mt_of(M), group, kc_blocks, swiglu ? 2 : 1).total;
}

int smallm_ctas_per_sm(int M, bool swiglu) {
    const int mt = mt_of(M);
    return (mt * (swiglu ? 2 : 1) <= 4) ? 2 : 1;
}

// Largest activation chunk (in k-blocks) that keeps one CTA's shared memory
// within the budget for the resident CTAs per SM.
int smallm_max_kc(int M, int group, bool swiglu) {
    const size_t budget = smallm_ctas_per_sm(M, swiglu) == 2 ? 112 * 1024 : 220 * 1024;
    int kc = 1;
    while (kc < 1024 && smallm_smem_bytes(M, group, swiglu, kc + 1) <= budget) ++kc;
    return kc;
}

cudaError_t launch_smallm(const SmallMParams &p, int group, bool swiglu, cudaStream_t s) {
    return swiglu ? launch_group<true>(p, group, s) : launch_group<false>(p, group, s);
}

}  // namespace w4a16
