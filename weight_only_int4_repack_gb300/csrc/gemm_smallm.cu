// Small-M W4A16 GEMM (decode / verify shapes, M <= 64): a weight-streaming kernel.
//
// At small M the GEMM is bound by reading the int4 weights once from HBM. The
// MatMulNBits Marlin pull request (github.com/justinchuby/onnx-genai pull 960,
// "P2 -- widen the win: split-K" and "Small-M split-K retune") found small M
// occupancy-bound and split the K range over more CTAs, reducing fp32 partials
// in a fixed order. This kernel keeps those two ideas and re-designs the rest
// for sm_103a:
//   * one CTA = one 128-row tile (eight 16-row sub-tiles) x one K range. In the
//     repacked layout four k-blocks of those sub-tiles are one regular 3-D box,
//     so a producer warp streams the range through a shared-memory ring with one
//     16 KB TMA copy per stage. The stream starts once the CTA's scales and zero
//     points have landed: they gate every group's flush, and issuing weights
//     earlier measured slower. The K split is chosen per shape so that the
//     busiest SM streams as few weight bytes as possible;
//   * consumer warps own one or two 16-row sub-tiles; a lane reads one 16-byte
//     slot per sub-tile and block (a conflict-free 128-bit shared load) whose
//     four words are mma.sync.m16n8k16 A fragments for four k16 steps; the
//     tokens are the n=8 operand and accumulation is fp32;
//   * dequantisation is 5 integer ops per 8 weights: OR-ing a nibble into the
//     mantissa of fp16 1024 gives exactly 1024 + q (bits 0-3) or 1024 + 16 q
//     (bits 4-7); in this layout the x16 form always belongs to the fragment's
//     second row (g+8). Per group and row the MMA gives acc_g = sum (1024 + f q) a
//     with f in {1, 16}, and
//         sum_g s_g sum (q - zp_g) a = sum_g (s_g/f) acc_g - sum_g (s_g/f)(1024 + f zp_g) A_g
//     where A_g is the group's activation sum. The first term is one fp32 FMA
//     per output and group (the pull request's "per-group scale AFTER the
//     tensor-core accumulate"); the second depends only on metadata and
//     activations and is subtracted once per staged chunk;
//   * the K split is a thread-block cluster: partial tiles are summed through
//     distributed shared memory in rank order (deterministic, no global scratch,
//     one launch).
// CUDA-core FMA would need M FMAs per weight; at M = 8 that is about 0.57 G FMA
// for K=5120, N=13824, more than the FP32 pipes finish in the HBM time of the
// weight stream, so the contraction runs on the tensor cores.
#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>

#include "ptx.cuh"
#include "w4a16_internal.h"

namespace w4a16 {
namespace {

constexpr int kPartStride = kTileRows + 4;          // floats per partial row (bank spread)
constexpr int kBPS = 4;                             // k-blocks per ring stage
constexpr int kStageSet = kTileRows * 32 * kBPS;   // 16 KB: one stage of one weight set
constexpr int kSubStage = kSubBytes * kBPS;         // 2 KB: one sub-tile's four k-blocks in a stage

// Ring stages of kStageSet bytes per weight set: 32 / 64 KB in flight per CTA.
constexpr int kStages = 2;

// Sub-tiles per consumer warp: two when the accumulators are small (shares the
// activation fragments and the per-block overhead), else one.
// A fused SwiGLU launch gives the gate and the up weight set CTAs of their own
// (one cluster = the K ranks of both sets), so every CTA streams one set.
template <int MT, bool SWIGLU>
struct Shape {
    static constexpr int SUBT = (MT <= 2) ? 2 : 1;
    static constexpr int CW = 8 / SUBT;             // consumer warps
    static constexpr int THREADS = CW * 32 + 32;    // + one producer warp
    static constexpr int STAGES = kStages;
    // CTAs per SM the register budget is sized for: fewer when the accumulators
    // grow, so that they stay in registers (measured at K=5120 N=13824: M=9
    // 16.4 vs 19.5 us, M=16 18.2 vs 20.3, M=32 32.6 vs 37.3 against the budget
    // of one token tile, which spilled).
    static constexpr int MINB = MT == 1 ? 4 : (MT == 2 ? 3 : 1);
};

// Compile-time loop: f(std::integral_constant<int, I>) for I in [B, E). Register
// arrays indexed by the constant stay in registers.
template <int B, int E, typename F>
__device__ __forceinline__ void static_for(F &&f) {
    if constexpr (B < E) {
        f(std::integral_constant<int, B>{});
        static_for<B + 1, E>(f);
    }
}

// (x & MASK) | 0x64006400 in one lop3: nibbles OR-ed into the mantissa of fp16 1024.
template <uint32_t MASK>
__device__ __forceinline__ uint32_t lop_or(uint32_t x) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(x), "n"(MASK), "n"(0x64006400));
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

// Shared-memory plan of one CTA (byte offsets from the dynamic base). The
// activation rows are the M token rows plus one zero row that padding tokens of
// the last 8-token tile read from.
struct SmemPlan {
    int a_stride, ng;
    size_t a_off, meta_off, gsum_off, bar_off, total;
};

__host__ __device__ inline SmemPlan make_plan(int M, int MT, int group, int kc, int stages) {
    SmemPlan p;
    p.a_off = (size_t)stages * kStageSet;          // the weight ring comes first
    p.a_stride = kc * kKBlock + 16;                 // +32 bytes per row: conflict-free fragment loads
    p.ng = (kc * kKBlock + group - 1) / group;      // groups of a chunk (chunks start on a group)
    p.meta_off = p.a_off + (size_t)(M + 1) * p.a_stride * 2;
    p.gsum_off = p.meta_off + (size_t)kTileRows * p.ng * 8;  // meta: float2 (s / f, (s / f)(1024 + f zp))
    const size_t main_end = p.gsum_off + (size_t)p.ng * 8 * MT * 4;  // float [ng][8 MT] group activation sums
    const size_t part_end = (size_t)8 * MT * kPartStride * 4;  // overlays the ring after use
    const size_t end = main_end > part_end ? main_end : part_end;
    p.bar_off = (end + 15) / 16 * 16;
    p.total = p.bar_off + (size_t)(2 * stages + 2) * 8;  // full[], empty[], activation barrier, abort
    return p;
}

template <int GROUP, int MT, bool SWIGLU>
__global__ void __launch_bounds__(Shape<MT, SWIGLU>::THREADS, Shape<MT, SWIGLU>::MINB)
    smallm_kernel(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                  const SmallMParams p) {
    using Sh = Shape<MT, SWIGLU>;
    constexpr int SUBT = Sh::SUBT, CW = Sh::CW, STAGES = Sh::STAGES;
    constexpr int NC = CW * 32;                            // consumer threads
    constexpr int SPG = GROUP / 16;                        // k16 steps per group
    constexpr int BPG = GROUP > kKBlock ? GROUP / kKBlock : 1;  // k-blocks per group (128: 2)
    static_assert((kBPS * 4) % SPG == 0, "a ring stage must hold whole groups");

    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    const int n0 = blockIdx.x * kTileRows;
    const int R = min(kTileRows, p.N - n0);
    const int nsub = R / kSubRows;
    const int S = p.split;                 // K ranks per weight set
    const int CS = SWIGLU ? 2 * S : S;     // cluster size: the K ranks of the gate, then of the up set
    const int crank = (CS > 1) ? (int)ptx::cluster_rank() : 0;
    const int set = SWIGLU ? crank / S : 0;  // weight set this CTA streams (SwiGLU: 0 gate, 1 up)
    const int rank = crank % S;
    // K ranges in whole groups, so that a group never straddles two ranks.
    const int nu = p.K / kKBlock / BPG;
    const int b_begin = (int)((long long)nu * rank / S) * BPG;
    const int b_end = (int)((long long)nu * (rank + 1) / S) * BPG;
    const int nstage = (b_end - b_begin + kBPS - 1) / kBPS;
    const int kc = p.kc_blocks;  // a multiple of kBPS unless it covers the whole range
    const SmemPlan plan = make_plan(p.M, MT, GROUP, kc, STAGES);

    uint64_t *full = reinterpret_cast<uint64_t *>(smem + plan.bar_off);
    uint64_t *empty = full + STAGES;
    uint64_t *abar = empty + STAGES;  // activation chunk landed
    volatile int *abort_flag = reinterpret_cast<volatile int *>(abar + 1);
    volatile int *a0_flag = abort_flag + 1;  // the producer issued the first activation chunk
    __half *sA = reinterpret_cast<__half *>(smem + plan.a_off);
    // Activation chunks: the producer issues the first, consumer thread 0 each later
    // one, only after it has seen the previous chunk land (one pending phase at
    // most). Thread 0 counts the chunk phases it has seen and the last chunk it
    // issued, so that after an abort it can wait for the one still in flight.
    int a_seen = 0, a_last = -1;

    // Activations [M][c0*64, c1*64) of a chunk: one bulk copy per token row.
    auto issue_activations = [&](int c0, int c1) {
        const uint32_t row_bytes = (uint32_t)(c1 - c0) * kKBlock * 2u;
        ptx::mbar_arrive_expect_tx(abar, (uint32_t)p.M * row_bytes);
        for (int m = 0; m < p.M; ++m)
            ptx::bulk_g2s(sA + (size_t)m * plan.a_stride, p.A + (size_t)m * p.K + (size_t)c0 * kKBlock, row_bytes,
                          abar);
    };
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], CW);
        }
        ptx::mbar_init(abar, 1);
        *abort_flag = 0;
        *a0_flag = 0;
        ptx::mbar_init_fence();
    }
    // Metadata of the first chunk, first batch of 8 groups per row: the loads are
    // issued before the barrier that releases the weight stream, so they are
    // ahead of it in the memory system (they are latency-critical, it is not).
    // In the common format (fp16 scales, G % 8 == 0) the raw words are kept and
    // converted after the barrier, so that no thread waits for them there and the
    // copies start at once.
    constexpr int RPT = (kTileRows + NC - 1) / NC;  // metadata rows per consumer thread
    const int zpstride = (p.G + 1) / 2;
    constexpr int PREB = RPT == 1 ? 2 : 1;  // prefetched batches of 8 groups
    const bool raw_meta = !p.scale_f32 && (p.G & 7) == 0;
    float pre_s[RPT][PREB][8];
    uint32_t pre_z[RPT][PREB][8];
    uint4 pre_x[RPT][PREB];       // raw fp16 scales of a batch (common format)
    uint32_t pre_zw[RPT][PREB];   // raw zero-point bytes of a batch (common format)
    // One batch = the 8 groups gbase .. gbase+7 of one row (gbase a multiple of 8);
    // groups outside [lo, hi) are not needed. fp16 scales in rows that start 16-byte
    // aligned (G % 8 == 0) come from one 16-byte load, their zero points from one
    // 4-byte load; other formats load each group.
    // Selected field by field: a runtime index into the parameter array would copy it to the stack.
    const void *const set_scales = set ? p.w[1].scales : p.w[0].scales;
    const uint8_t *const set_zp = set ? p.w[1].zp : p.w[0].zp;
    auto load_meta_batch = [&](int row, int gbase, int lo, int hi, float (&sv)[8], uint32_t (&zb)[8]) {
        const int n = n0 + row;
        const uint8_t *zrow = set_zp ? set_zp + (size_t)n * zpstride : nullptr;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            sv[u] = 0.f;
            zb[u] = 0x88u;
        }
        // No load for a window that holds none of the needed groups (it may lie
        // past the end of the row); a window that does ends inside its row.
        if (row >= R || gbase >= hi || gbase + 8 <= lo) return;
        if (!p.scale_f32 && (p.G & 7) == 0) {
            const uint4 x = __ldg(reinterpret_cast<const uint4 *>(
                reinterpret_cast<const unsigned short *>(set_scales) + (size_t)n * p.G + gbase));
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
            const uint32_t zw = zrow ? __ldg(reinterpret_cast<const unsigned int *>(zrow + gbase / 2)) : 0x88888888u;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                sv[u] = __half2float(__ushort_as_half((unsigned short)(xs[u >> 1] >> (16 * (u & 1)))));
                zb[u] = (zw >> (8 * (u >> 1))) & 0xFFu;
            }
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int grp = gbase + u;
                if (grp >= lo && grp < hi) {
                    const size_t si = (size_t)n * p.G + grp;
                    sv[u] = p.scale_f32 ? __ldg(reinterpret_cast<const float *>(set_scales) + si)
                                        : __half2float(__ldg(reinterpret_cast<const __half *>(set_scales) + si));
                    if (zrow) zb[u] = __ldg(zrow + (grp >> 1));
                }
            }
        }
    };
    // Raw words of one batch (common format); a window that holds none of the
    // needed groups is not loaded (it may lie past the end of the row).
    auto load_raw_batch = [&](int row, int gbase, int lo, int hi, uint4 &x, uint32_t &zw) {
        x = make_uint4(0u, 0u, 0u, 0u);
        zw = 0x88888888u;
        if (row >= R || gbase >= hi || gbase + 8 <= lo) return;
        const int n = n0 + row;
        x = __ldg(reinterpret_cast<const uint4 *>(reinterpret_cast<const unsigned short *>(set_scales) +
                                                  (size_t)n * p.G + gbase));
        if (set_zp) zw = __ldg(reinterpret_cast<const unsigned int *>(set_zp + (size_t)n * zpstride + gbase / 2));
    };
    const int grp_first0 = (b_begin * kKBlock) / GROUP;
    const int ng_first0 = ((min(b_begin + kc, b_end) - b_begin) * kKBlock) / GROUP;
    if (warp < CW) {
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int rs = tid + NC * r;
            if (rs < kTileRows) {
#pragma unroll
                for (int bt = 0; bt < PREB; ++bt) {
                    const int gbase = (grp_first0 & ~7) + 8 * bt;
                    if (raw_meta)
                        load_raw_batch(rs, gbase, grp_first0, grp_first0 + ng_first0, pre_x[r][bt], pre_zw[r][bt]);
                    else
                        load_meta_batch(rs, gbase, grp_first0, grp_first0 + ng_first0, pre_s[r][bt], pre_z[r][bt]);
                }
            }
        }
    }
    __syncthreads();
    ptx::grid_dep_launch();

    if (warp == CW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            // A may be the previous kernel's output: it is read only after the
            // wait on that kernel. Weights, scales and zero points are not, so as
            // a programmatic dependent the first ring stages go out before it.
            const int pre = p.overlap ? min(STAGES, nstage) : 0;
            bool a_issued = false;
            auto start_activations = [&]() {
                ptx::grid_dep_wait();
                *a0_flag = 1;
                issue_activations(b_begin, min(b_begin + kc, b_end));
                a_issued = true;
            };
            if (pre == 0) start_activations();
            const uint64_t stream_policy = ptx::policy_evict_first();
            const CUtensorMap *tm_w = set ? &tm_w1 : &tm_w0;
            ptx::prefetch_tmap(tm_w);
            int st = 0;
            for (; st < nstage; ++st) {
                const int s = st % STAGES;
                const uint32_t ph = (uint32_t)(st / STAGES) & 1u;
                if (st == pre && !a_issued) start_activations();
                if (!ptx::mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.err, p.wait_ns)) break;
                const int b0 = b_begin + st * kBPS;
                // One box: kBPS k-blocks of the tile's eight sub-tiles (sub-tiles past N
                // and k-blocks past K read as zero), [sub-tile][k-block][512 bytes].
                ptx::mbar_arrive_expect_tx(&full[s], kStageSet);
                unsigned char *dst = smem + (size_t)s * kStageSet;
                ptx::tma_load_3d_hint(dst, tm_w, 0, b0, n0 / kSubRows, &full[s], stream_policy);
            }
            if (!a_issued && !*abort_flag) start_activations();
            if (*abort_flag) {
                // Let the copies already issued land before the CTA can exit.
                volatile int no_abort = 0;
                for (int s = 0; s < STAGES && s < st; ++s) {
                    const int last = s + ((st - 1 - s) / STAGES) * STAGES;
                    ptx::mbar_wait(&full[s], (uint32_t)(last / STAGES) & 1u, &no_abort, nullptr, 200000000ull);
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ consumers
        const int g = lane >> 2, t = lane & 3;
        const int slot = 4 * g + ((t + (g >> 1)) & 3);  // lane slot of fragment (g, t)
        for (int i = tid; i < plan.a_stride; i += NC) sA[(size_t)p.M * plan.a_stride + i] = __float2half(0.f);
        bool sub_ok[SUBT];
#pragma unroll
        for (int u = 0; u < SUBT; ++u) sub_ok[u] = warp * SUBT + u < nsub;
        // Shared-memory row of token 8*mt + g (padding tokens read the zero row).
        int arow[MT];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) arow[mt] = min(8 * mt + g, p.M) * plan.a_stride;
        const float2 *meta0 = reinterpret_cast<const float2 *>(smem + plan.meta_off);
        int mrow[SUBT][2];
#pragma unroll
        for (int u = 0; u < SUBT; ++u) {
            const int rg = (warp * SUBT + u) * kSubRows + g;
            mrow[u][0] = rg * plan.ng;
            mrow[u][1] = (rg + 8) * plan.ng;
        }

        float acc[SUBT][MT][4];
#pragma unroll
        for (int u = 0; u < SUBT; ++u)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[u][mt][i] = 0.f;

        bool aborted = false;
        for (int c0 = b_begin; c0 < b_end; c0 += kc) {
            const int c1 = min(c0 + kc, b_end);
            const int grp0 = (c0 * kKBlock) / GROUP;
            const int ng = ((c1 - c0) * kKBlock) / GROUP;
            ptx::named_bar_sync(1, NC);  // previous chunk consumed
            const int chunk_idx = (c0 - b_begin) / kc;
            if (tid == 0 && c0 != b_begin && !aborted && !*abort_flag) {
                // Generic reads of sA (previous chunk) before the async writes.
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue_activations(c0, c1);
                a_last = chunk_idx;
            }
            // Per row and group: (s / f, (s / f)(1024 + f zp)), f = 16 for the second
            // row of each 16-row fragment block. One row per thread, loads batched.
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const int rs = tid + NC * r;
                if (rs >= kTileRows) continue;
                const int row = rs;
                if (row >= R) continue;
                float2 *meta = reinterpret_cast<float2 *>(smem + plan.meta_off) + (size_t)row * plan.ng;
                const bool hi_row = (row >> 3) & 1;
                const float f = hi_row ? 16.f : 1.f, inv_f = hi_row ? 0.0625f : 1.f;
                const int gbase0 = grp0 & ~7;  // batches start on 8-group boundaries
                for (int gb = gbase0; gb < grp0 + ng; gb += 8) {
                    const int bt = (gb - gbase0) >> 3;
                    float sv[8];
                    uint32_t zb[8];
                    if (c0 == b_begin && bt < PREB && raw_meta) {
                        const uint4 x = bt == 0 ? pre_x[r][0] : pre_x[r][PREB - 1];
                        const uint32_t zw = bt == 0 ? pre_zw[r][0] : pre_zw[r][PREB - 1];
                        const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            sv[u] = __half2float(__ushort_as_half((unsigned short)(xs[u >> 1] >> (16 * (u & 1)))));
                            zb[u] = (zw >> (8 * (u >> 1))) & 0xFFu;
                        }
                    } else if (c0 == b_begin && bt < PREB) {
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            sv[u] = bt == 0 ? pre_s[r][0][u] : pre_s[r][PREB - 1][u];
                            zb[u] = bt == 0 ? pre_z[r][0][u] : pre_z[r][PREB - 1][u];
                        }
                    } else {
                        load_meta_batch(rs, gb, grp0, grp0 + ng, sv, zb);
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int grp = gb + u, gi = grp - grp0;
                        if (gi >= 0 && gi < ng) {
                            const float zv = (float)((grp & 1) ? (zb[u] >> 4) : (zb[u] & 0xFu));
                            const float sf = sv[u] * inv_f;  // exact: f is a power of two
                            meta[gi] = make_float2(sf, sf * (1024.f + f * zv));
                        }
                    }
                }
            }
            if (!aborted && !ptx::mbar_wait(abar, (uint32_t)chunk_idx & 1u, abort_flag, p.err, p.wait_ns)) aborted = true;
            if (!aborted) a_seen = chunk_idx + 1;
            // Group activation sums A_g[token] of this chunk (fp32 over the fp16
            // values), one (group, token) per thread with independent loads.
            {
                float *gs = reinterpret_cast<float *>(smem + plan.gsum_off);
                for (int i = tid; i < ng * 8 * MT; i += NC) {
                    const int gi = i / (8 * MT), m = i % (8 * MT);
                    float v0 = 0.f, v1 = 0.f;
                    if (m < p.M && !aborted) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(sA + (size_t)m * plan.a_stride + gi * GROUP);
#pragma unroll
                        for (int q = 0; q < GROUP / 8; ++q) {
                            const uint4 x = src[q];
                            const __half2 *h = reinterpret_cast<const __half2 *>(&x);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f2 = __half22float2(h[e]);
                                v0 += f2.x;
                                v1 += f2.y;
                            }
                        }
                    }
                    gs[i] = v0 + v1;
                }
            }
            ptx::named_bar_sync(1, NC);

            float accg[SUBT][MT][4];  // partial sum of the current group
            const int st0 = (c0 - b_begin) / kBPS, st1 = (c1 - b_begin + kBPS - 1) / kBPS;
            for (int st = st0; st < st1; ++st) {
                const int s = st % STAGES;
                const uint32_t ph = (uint32_t)(st / STAGES) & 1u;
                if (!aborted && !ptx::mbar_wait(&full[s], ph, abort_flag, p.err, p.wait_ns)) aborted = true;
                if (aborted) continue;
                const int bs = b_begin + st * kBPS;  // first k-block of the stage
                // Per-stage bases: every offset below them is a compile-time constant
                // (weights sit in fixed 4 KB block slots, stages start on a group).
                const unsigned char *wbase =
                    smem + (size_t)s * kStageSet + (warp * SUBT) * kSubStage + slot * 16;
                const __half *abase = sA + (bs - c0) * kKBlock + 4 * t;
                const float2 *mbase = meta0 + ((bs - c0) * kKBlock) / GROUP;
                auto run_stage = [&](auto nbc) {
                    constexpr int NB = decltype(nbc)::value;
                    static_for<0, NB>([&](auto ic) {
                        constexpr int i = decltype(ic)::value;
                        uint4 wv[SUBT];
                        static_for<0, SUBT>([&](auto uc) {
                            constexpr int u = decltype(uc)::value;
                            wv[u] = *reinterpret_cast<const uint4 *>(wbase + u * kSubStage + i * kSubBytes);
                        });
                        static_for<0, 4>([&](auto jc) {
                            constexpr int j = decltype(jc)::value;
                            constexpr int step = i * 4 + j;  // k16 step within the stage
                            // Activation fragment of each token tile: k = 16j + 4t .. +3.
                            uint32_t bfr[MT][2];
#pragma unroll
                            for (int mt = 0; mt < MT; ++mt) {
                                const uint2 v =
                                    *reinterpret_cast<const uint2 *>(abase + arow[mt] + i * kKBlock + 16 * j);
                                bfr[mt][0] = v.x;
                                bfr[mt][1] = v.y;
                            }
                            static_for<0, SUBT>([&](auto uc) {
                                constexpr int u = decltype(uc)::value;
                                const uint32_t word = j == 0 ? wv[u].x : j == 1 ? wv[u].y : j == 2 ? wv[u].z : wv[u].w;
                                const uint32_t w8 = word >> 8;
                                uint32_t a[4];
                                a[0] = lop_or<0x000F000Fu>(word);  // row g,   k 4t+0/1: 1024 + q
                                a[1] = lop_or<0x00F000F0u>(word);  // row g+8, k 4t+0/1: 1024 + 16 q
                                a[2] = lop_or<0x000F000Fu>(w8);    // row g,   k 4t+2/3
                                a[3] = lop_or<0x00F000F0u>(w8);    // row g+8, k 4t+2/3
#pragma unroll
                                for (int mt = 0; mt < MT; ++mt) {
                                    if constexpr (step % SPG == 0) {
                                        const float z4[4] = {0.f, 0.f, 0.f, 0.f};
                                        mma_16816(accg[u][mt], a, bfr[mt][0], bfr[mt][1], z4);
                                    } else {
                                        mma_16816(accg[u][mt], a, bfr[mt][0], bfr[mt][1], accg[u][mt]);
                                    }
                                }
                            });
                            if constexpr (step % SPG == SPG - 1) {
                                // Group complete: acc += (s / f) * acc_g.
                                constexpr int gs = (i * kKBlock + 16 * j) / GROUP;  // group within the stage
                                static_for<0, SUBT>([&](auto uc) {
                                    constexpr int u = decltype(uc)::value;
                                    const float s0 = mbase[mrow[u][0] + gs].x;
                                    const float s1 = mbase[mrow[u][1] + gs].x;
#pragma unroll
                                    for (int mt = 0; mt < MT; ++mt) {
                                        float *ac = acc[u][mt];
                                        const float *ag = accg[u][mt];
                                        ac[0] = fmaf(s0, ag[0], ac[0]);
                                        ac[1] = fmaf(s0, ag[1], ac[1]);
                                        ac[2] = fmaf(s1, ag[2], ac[2]);
                                        ac[3] = fmaf(s1, ag[3], ac[3]);
                                    }
                                });
                            }
                        });
                    });
                };
                const int nb = min(kBPS, c1 - bs);  // blocks of this stage (whole groups)
                if (nb == kBPS) {
                    run_stage(std::integral_constant<int, kBPS>{});
                } else if constexpr (BPG == 1) {
                    if (nb == 1) run_stage(std::integral_constant<int, 1>{});
                    else if (nb == 2) run_stage(std::integral_constant<int, 2>{});
                    else run_stage(std::integral_constant<int, 3>{});
                } else {
                    run_stage(std::integral_constant<int, 2>{});  // 128-wide groups: two blocks
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&empty[s]);
            }
            // Offset and zero-point term of this chunk: acc -= sum_g (s/f)(1024 + f zp) A_g.
            {
                const float *gsum = reinterpret_cast<const float *>(smem + plan.gsum_off);
                for (int gi = 0; gi < ng; ++gi) {
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        const float2 ag = *reinterpret_cast<const float2 *>(gsum + gi * 8 * MT + 8 * mt + 2 * t);
#pragma unroll
                        for (int u = 0; u < SUBT; ++u) {
                            const float c0v = meta0[mrow[u][0] + gi].y;
                            const float c1v = meta0[mrow[u][1] + gi].y;
                            float *ac = acc[u][mt];
                            ac[0] = fmaf(-c0v, ag.x, ac[0]);
                            ac[1] = fmaf(-c0v, ag.y, ac[1]);
                            ac[2] = fmaf(-c1v, ag.x, ac[2]);
                            ac[3] = fmaf(-c1v, ag.y, ac[3]);
                        }
                    }
                }
            }
        }

        // Partial tile -> shared memory as [token][row]; it overlays the ring,
        // which every consumer warp has finished with (all copies have landed).
        ptx::named_bar_sync(1, NC);
        float *P = reinterpret_cast<float *>(smem);
#pragma unroll
        for (int u = 0; u < SUBT; ++u) {
            if (!sub_ok[u]) continue;
            const int rg = (warp * SUBT + u) * kSubRows + g;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const int m0 = 8 * mt + 2 * t;
                P[(size_t)m0 * kPartStride + rg] = acc[u][mt][0];
                P[(size_t)(m0 + 1) * kPartStride + rg] = acc[u][mt][1];
                P[(size_t)m0 * kPartStride + rg + 8] = acc[u][mt][2];
                P[(size_t)(m0 + 1) * kPartStride + rg + 8] = acc[u][mt][3];
            }
        }
    }

    if (CS > 1) ptx::cluster_sync(); else __syncthreads();
    if (tid == 0) {
        // After an abort an activation chunk may still be in flight: the last one
        // issued, if thread 0 has not seen it land. Wait (bounded) before exit.
        const int last = a_last >= 0 ? a_last : (*a0_flag ? 0 : -1);
        if (last >= a_seen) {
            volatile int no_abort = 0;
            ptx::mbar_wait(abar, (uint32_t)last & 1u, &no_abort, nullptr, 200000000ull);
        }
    }
    ptx::grid_dep_wait();  // Y may still be in use by the previous kernel

    // Cluster rank r finalises rows [r*R/CS, (r+1)*R/CS): each set's partials of its
    // K ranks summed in rank order, then (SwiGLU) silu(gate) * up.
    {
        constexpr int NSET = SWIGLU ? 2 : 1;
        const float *P = reinterpret_cast<const float *>(smem);
        const int lo = (int)((long long)R * crank / CS), hi = (int)((long long)R * (crank + 1) / CS);
        const int nr = hi - lo;
        for (int i = tid; i < p.M * nr; i += Sh::THREADS) {
            const int m = i / nr, row = lo + i % nr;
            const float *src = P + (size_t)m * kPartStride + row;
            float v[NSET];
#pragma unroll
            for (int w = 0; w < NSET; ++w) {
                if (CS > 1) {
                    float part[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        part[q] = q < S ? ptx::ld_dsmem_f32(src, (uint32_t)(w * S + q)) : 0.f;
                    float sum = part[0];
#pragma unroll
                    for (int q = 1; q < 8; ++q)
                        if (q < S) sum += part[q];  // rank order: deterministic
                    v[w] = sum;
                } else {
                    v[w] = *src;
                }
            }
            float y = v[0];
            if constexpr (SWIGLU) y = silu_f32(v[0]) * v[NSET - 1];
            p.Y[(size_t)m * p.N + n0 + row] = __float2half_rn(y);
        }
    }
    if (CS > 1) ptx::cluster_sync();  // keep shared memory alive until every peer has read it
}

constexpr int kMaxDynSmem = 227 * 1024;

// Raise the kernel's dynamic shared-memory limit once per device.
template <int GROUP, int MT, bool SWIGLU>
cudaError_t configure() {
    return ensure_max_dyn_smem(reinterpret_cast<const void *>(smallm_kernel<GROUP, MT, SWIGLU>), kMaxDynSmem);
}

// CTAs of a (1 x cs) cluster launch that the device keeps resident at once.
template <int GROUP, int MT, bool SWIGLU>
int occupancy(size_t smem, int cs) {
    if (configure<GROUP, MT, SWIGLU>() != cudaSuccess) return 0;
    int n = 0;
    if (cs <= 1) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, smallm_kernel<GROUP, MT, SWIGLU>,
                                                          Shape<MT, SWIGLU>::THREADS, smem) != cudaSuccess)
            return 0;
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        return n * sms;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1024, (unsigned)cs, 1);
    cfg.blockDim = dim3(Shape<MT, SWIGLU>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)cs;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, smallm_kernel<GROUP, MT, SWIGLU>, &cfg) != cudaSuccess) return 0;
    return n * cs;
}

template <int GROUP, int MT, bool SWIGLU>
cudaError_t launch_one(const SmallMParams &p, cudaStream_t s) {
    const size_t smem = make_plan(p.M, MT, GROUP, p.kc_blocks, Shape<MT, SWIGLU>::STAGES).total;
    auto kern = smallm_kernel<GROUP, MT, SWIGLU>;
    cudaError_t e = configure<GROUP, MT, SWIGLU>();
    if (e != cudaSuccess) return e;
    const int cs = SWIGLU ? 2 * p.split : p.split;  // cluster: the K ranks of each weight set
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.N + kTileRows - 1) / kTileRows), (unsigned)cs, 1);
    cfg.blockDim = dim3(Shape<MT, SWIGLU>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (cs > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = (unsigned)cs;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (p.overlap) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    CUtensorMap m0, m1;
    if (!tmap_weights(&m0, p.w[0].q_rep, p.N, p.K, kBPS, kTileRows / kSubRows)) return cudaErrorInvalidValue;
    if (!tmap_weights(&m1, p.w[SWIGLU ? 1 : 0].q_rep, p.N, p.K, kBPS, kTileRows / kSubRows))
        return cudaErrorInvalidValue;
    return cudaLaunchKernelEx(&cfg, kern, m0, m1, p);
}

template <int GROUP, bool SWIGLU>
int occupancy_mt(int M, size_t smem, int cs) {
    const int mt = (M + 7) / 8;
    if (mt <= 1) return occupancy<GROUP, 1, SWIGLU>(smem, cs);
    if (mt <= 2) return occupancy<GROUP, 2, SWIGLU>(smem, cs);
    if (mt <= 4) return occupancy<GROUP, 4, SWIGLU>(smem, cs);
    return occupancy<GROUP, 8, SWIGLU>(smem, cs);
}

template <bool SWIGLU>
int occupancy_group(int M, int group, size_t smem, int cs) {
    switch (group) {
        case 16: return occupancy_mt<16, SWIGLU>(M, smem, cs);
        case 32: return occupancy_mt<32, SWIGLU>(M, smem, cs);
        case 64: return occupancy_mt<64, SWIGLU>(M, smem, cs);
        default: return occupancy_mt<128, SWIGLU>(M, smem, cs);
    }
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

int threads_of(int M, bool swiglu) {
    (void)swiglu;  // a SwiGLU CTA streams one weight set, as a plain one does
    const int subt = (mt_of(M) <= 2) ? 2 : 1;
    return (8 / subt) * 32 + 32;
}

}  // namespace

size_t smallm_smem_bytes(int M, int group, bool swiglu, int kc_blocks) {
    (void)swiglu;
    return make_plan(M, mt_of(M), group, kc_blocks, kStages).total;
}

int smallm_threads(int M, bool swiglu) { return threads_of(M, swiglu); }

// Split (cluster size) and activation chunk for one shape. Among plans whose
// grid is resident at once (one wave), the choice minimises the weight blocks
// the busiest SM streams (CTAs per SM, rounded up, x blocks per CTA): measured
// on GB300 at M=8 K=5120 N=13824, split 4 (432 CTAs, at most 3 per SM) beats
// split 5 (540 CTAs, up to 4 per SM) by 9%. Ties go to the larger grid (more
// bytes in flight), then to fewer activation chunks. Splits that give every rank
// the same number of groups come first: at K=13824 N=5120 (108 groups) split 6
// ran in 15.4 us against 22.9 for split 7, which the block count prefers. Without a one-wave plan, a
// time model decides: waves x (blocks an SM streams per wave + a fixed cost per
// CTA). A forced split only picks the chunk. SwiGLU launches a cluster of
// 2 x split CTAs (gate and up ranks), so split <= 4.
// The fixed cost of one CTA (start, metadata, split-K reduction) in k-blocks of
// streaming. At M=32 K=5120 N=13824 fused SwiGLU (CTAs of one per SM) it makes
// split 2 (three waves of half ranges) win over split 1 (two waves of full ranges).
constexpr int kFixedBlocks = 5;

SmallMPlan smallm_plan(int M, int N, int K, int group, bool swiglu, int split_k, int sm_count) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int, bool, int, int>, SmallMPlan> cache;
    const auto key = std::make_tuple(M, N, K, group, swiglu, split_k, sm_count);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    const int bpg = group > kKBlock ? group / kKBlock : 1;  // k-blocks per group
    const int nu = K / kKBlock / bpg;                       // K split unit: whole groups
    const int n_tiles = (N + kTileRows - 1) / kTileRows;
    SmallMPlan best{};
    long long best_score = -1;              // multi-wave plans (used only if no one-wave plan): cost
    SmallMPlan best1{};
    long long best1_work = 0, best1_grid = 0;
    bool best1_even = false;
    int best1_chunks = 0;
    const int hi = split_k > 0 ? split_k : (swiglu ? 4 : 8);
    const int lo = split_k > 0 ? split_k : 1;
    for (int split = hi; split >= lo; --split) {
        if (split > nu) continue;
        const int per_rank = (nu + split - 1) / split * bpg;
        const int pf = kBPS;  // chunk boundaries stay on ring-stage boundaries
        int prev_kc = -1;
        for (int chunks = 1; chunks <= 8; ++chunks) {
            int kc = (per_rank + chunks - 1) / chunks;
            if (chunks > 1) kc = (kc + pf - 1) / pf * pf;
            if (kc >= per_rank && chunks > 1) continue;
            if (kc == prev_kc) continue;
            prev_kc = kc;
            const size_t smem = smallm_smem_bytes(M, group, swiglu, kc);
            if (smem > (size_t)kMaxDynSmem) continue;
            const int cs = swiglu ? 2 * split : split;  // CTAs per cluster
            if (cs > 8) continue;
            const int resident = swiglu ? occupancy_group<true>(M, group, smem, cs)
                                        : occupancy_group<false>(M, group, smem, cs);
            if (resident <= 0) continue;
            const int occ = (resident + sm_count - 1) / sm_count;
            const long long grid = (long long)n_tiles * cs;
            const long long slots = resident;
            const long long waves = (grid + slots - 1) / slots;
            if (waves == 1) {
                const long long work = (grid + sm_count - 1) / sm_count * per_rank;  // busiest SM
                const bool even = nu % split == 0;  // every rank the same number of groups
                const bool better = best1.split == 0 || (even && !best1_even) ||
                                    (even == best1_even &&
                                     (work < best1_work ||
                                      (work == best1_work && (grid > best1_grid ||
                                                              (grid == best1_grid && chunks < best1_chunks)))));
                if (better) {
                    best1 = SmallMPlan{split, (int)kc, (int)smem, occ};
                    best1_work = work;
                    best1_grid = grid;
                    best1_chunks = chunks;
                    best1_even = even;
                }
                break;  // more chunks only shrink the chunk further
            }
            // Time model in k-blocks: every wave streams its CTAs' ranges (the
            // CTAs sharing an SM share its stream) plus a fixed start and
            // reduction cost per CTA; extra activation chunks cost a little more.
            const long long per_sm = (slots + sm_count - 1) / sm_count;
            const long long cost = waves * (per_sm * per_rank + kFixedBlocks) + (chunks - 1) * 2;
            if (best_score < 0 || cost < best_score) {
                best_score = cost;
                best = SmallMPlan{split, (int)kc, (int)smem, occ};
            }
        }
    }
    if (best1.split != 0) best = best1;
    if (best.split == 0) {
        // Nothing fit: the smallest chunk that is still whole ring stages and whole groups.
        const int kc = std::min(K / kKBlock, std::max(kBPS, bpg));
        best = SmallMPlan{1, kc, (int)smallm_smem_bytes(M, group, swiglu, kc), 1};
    }
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = best;
    return best;
}

cudaError_t launch_smallm(const SmallMParams &p, int group, bool swiglu, cudaStream_t s) {
    return swiglu ? launch_group<true>(p, group, s) : launch_group<false>(p, group, s);
}

}  // namespace w4a16
