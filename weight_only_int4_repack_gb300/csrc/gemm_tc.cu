// Large-M W4A16 GEMM on the 5th-generation tensor cores (tcgen05, tensor memory).
//
// The MatMulNBits Marlin pull request (github.com/justinchuby/onnx-genai pull
// 960, "What's landed") runs an SM80 mma.sync kernel for every M > 1. On sm_103a
// the contraction at large M belongs on tcgen05, so this kernel is new:
//   * roles are swapped: the dequantised weights are the MMA's A operand (M = 128
//     weight rows per tile) held in tensor memory, and the activations are the B
//     operand (N = T tokens, 16..256) staged by TMA with the 128-byte swizzle;
//     D = W . A^T accumulates in fp32 in tensor memory;
//   * a producer warp issues, per 64-k block, one TMA box of activations and one
//     3-D TMA box of the weight chunk (eight 512-byte sub-tile pieces of the
//     repacked layout, 4 KB) into a ring of shared-memory stages;
//   * three groups of four dequant warps (one warp per tensor-memory lane
//     quarter, one thread per weight row) take every third k-block: a thread
//     reads its row's nibbles from the chunk (conflict-free thanks to the
//     layout's lane-slot rotation), forms w = (q - zp) * s in fp16 (nibbles
//     OR-ed into the mantissa of 1024, one exact subtraction of 1024 + zp, one
//     multiply by the scale) and stores the block's 32 packed columns with one
//     tcgen05.st;
//   * the shared-memory ring of copies and the tensor-memory ring of A stages
//     advance together, one "empty" barrier per stage freeing both;
//   * one thread issues the four K=16 MMAs per block and commits them to the
//     stage's "empty" barrier; it issues every MMA of the CTA and each of its
//     barrier waits, MMAs and commits costs tens of nanoseconds, so it waits
//     only on the A stage, which the dequant warps fill after they have seen the
//     copies land, and commits once per block;
//     after the last block a commit releases the epilogue (the dequant warps),
//     which reads the accumulator with tcgen05.ld and stores fp16;
//   * fused SwiGLU keeps the plain GEMM's 256-token tile: a CTA owns 64 output
//     columns, and its 128 MMA rows are those 64 gate rows and the same 64 up
//     rows (two 2 KB halves of the repacked chunks), interleaved by 16 so that
//     each lane quarter holds the gate and the up rows of 16 columns; one
//     accumulator holds both, every dequantised weight still serves 256 tokens,
//     and the epilogue pairs lane l with lane l ^ 16 by a shuffle and stores
//     silu(gate) * up.
// Every mbarrier wait is bounded; on expiry the kernel records
// W4A16_ERR_TIMEOUT, drains what it issued, frees its tensor memory and returns.
#include <map>
#include <mutex>
#include <tuple>

#include "ptx.cuh"
#include "w4a16_internal.h"

namespace w4a16 {
namespace {

// Dequantisation: kDqParts warp groups (one warp per tensor-memory lane quarter
// each) take every kDqParts-th k-block, a thread converting all four k16 steps of
// its row, so that more warps hide each other's latencies. Both ring depths are
// multiples of kDqParts: then a group's next block in a ring slot is the slot's
// very next use, so its parity wait can never match a phase two uses old.
constexpr int kSPW = 4;                      // k16 steps of a block that one dequant thread converts
constexpr int kDqParts = 3;                  // dequant warp groups (= warps per lane quarter)
constexpr int kDqThreads = 128 * kDqParts;   // dequant / epilogue threads
constexpr int kThreads = 64 + kDqThreads;    // warp 0 producer, warp 1 MMA + TMEM, then dequant/epilogue
constexpr int kTmemCols = 512;
constexpr int kChunk = kTileRows * 32;  // 4 KB weight chunk per 64-k block
struct TcShape {
    static constexpr int NS = 1;        // one accumulator (SwiGLU pairs its rows inside it)
    static constexpr int TMAX = 256;    // tokens per tile (MMA N)
    static constexpr int STAGES = 6;    // shared-memory ring (TMA in flight)
    static constexpr int ASTAGES = 6;   // tensor-memory A stages: T + ASTAGES*32 <= 512
    static_assert(STAGES % kDqParts == 0 && ASTAGES % kDqParts == 0, "ring depths: multiples of the dequant groups");
    static_assert(STAGES == ASTAGES, "one barrier frees a shared-memory stage and its tensor-memory A stage");
};

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(ptx::smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16, one CTA.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on `bar` once every tcgen05 operation this thread issued so far is complete.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     ptx::smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[N]) {
    static_assert(N == 8 || N == 16 || N == 32, "8, 16 or 32 columns");
    if constexpr (N == 32) tmem_st32(taddr, r);
    else if constexpr (N == 16) tmem_st16(taddr, r);
    else tmem_st8(taddr, r);
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);          // start address
    d |= (uint64_t)1u << 16;                           // leading byte offset (unused for this layout)
    d |= (uint64_t)(1024u >> 4) << 32;                 // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1u << 46;                           // descriptor version for tcgen05
    d |= (uint64_t)2u << 61;                           // layout: 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (K-major), fp32 D, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_f16(int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// silu(x) = x / (1 + e^-x) with the hardware exponential and reciprocal intrinsics
// (relative error about 1e-6, far below the fp16 rounding of the output): the
// fused epilogue evaluates it for every output, unoverlapped with the MMAs.
__device__ __forceinline__ float silu_f32(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// Shared memory: [B stages (1024-aligned)] [W stages] [barriers] [tmem slot].
struct TcSmem {
    int T, stages, astages, ns;
    size_t b_stage, w_off, bar_off, total;
};
__host__ __device__ inline TcSmem tc_smem(int T, int stages, int astages, int ns) {
    TcSmem p;
    p.T = T;
    p.stages = stages;
    p.astages = astages;
    p.ns = ns;
    p.b_stage = (size_t)T * 128;  // T token rows x 64 fp16
    p.w_off = p.b_stage * stages;
    p.bar_off = p.w_off + (size_t)stages * ns * kChunk;
    p.total = p.bar_off + (size_t)(2 * stages + astages + 2) * 8 + 16;
    return p;
}

// Per-row metadata of k-block kb for the k16 steps j0 .. j0+kSPW-1: half2
// (1024 + zp) and half2 s (steps in one group share them).
template <int GROUP>
__device__ __forceinline__ void load_row_meta(const TcParams &p, const void *scales, const uint8_t *zp, int n, int kb,
                                              int j0, uint32_t (&zz)[kSPW], uint32_t (&ss)[kSPW]) {
#pragma unroll
    for (int jj = 0; jj < kSPW; ++jj) {
        if (jj > 0 && (16 * (j0 + jj)) / GROUP == (16 * (j0 + jj - 1)) / GROUP) {
            zz[jj] = zz[jj - 1];
            ss[jj] = ss[jj - 1];
            continue;
        }
        const int grp = (kb * kKBlock + 16 * (j0 + jj)) / GROUP;
        const size_t si = (size_t)n * p.G + grp;
        float s;
        if (p.scale_f32) s = __ldg(reinterpret_cast<const float *>(scales) + si);
        else s = __half2float(__ldg(reinterpret_cast<const __half *>(scales) + si));
        uint32_t z = 8;
        if (zp) {
            const uint8_t zb = __ldg(zp + (size_t)n * ((p.G + 1) / 2) + (grp >> 1));
            z = (grp & 1) ? (zb >> 4) : (zb & 0xFu);
        }
        const uint32_t zh = 0x6400u + z;  // fp16 bits of 1024 + zp
        zz[jj] = zh | (zh << 16);
        const uint32_t sh = (uint32_t)__half_as_ushort(__float2half_rn(s));
        ss[jj] = sh | (sh << 16);
    }
}

template <int GROUP, bool SWIGLU>
__global__ void __launch_bounds__(kThreads, 1)
    tc_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w0,
              const __grid_constant__ CUtensorMap tmap_w1, const TcParams p, int T) {
    using Sh = TcShape;
    constexpr int NS = Sh::NS, STAGES = Sh::STAGES, ASTAGES = Sh::ASTAGES;
    constexpr int COLS = SWIGLU ? 64 : kTileRows;  // output columns per CTA

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // The B stages need 1024-byte alignment (128-byte swizzle atoms).
    unsigned char *smem = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const TcSmem L = tc_smem(T, STAGES, ASTAGES, NS);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bar_off);  // TMA + bulk copy landed
    uint64_t *empty = full + STAGES;    // MMAs done with the stage (shared memory and A columns)
    uint64_t *afull = empty + STAGES;   // A stage written to tensor memory
    uint64_t *accfull = afull + ASTAGES;
    uint64_t *drain = accfull + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m0 = blockIdx.x * T;
    const int n0 = blockIdx.y * COLS;               // first output column
    const int R = min(COLS, p.N - n0);              // output columns of this CTA
    const int sub0 = n0 / kSubRows;                 // first 16-row sub-tile of those columns
    const int nkb = p.K / kKBlock;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < ASTAGES; ++s) ptx::mbar_init(&afull[s], kDqThreads / kDqParts);  // one warp group per block
        ptx::mbar_init(accfull, 1);
        ptx::mbar_init(drain, 1);
        *abort_flag = 0;
        ptx::mbar_init_fence();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Tensor-memory columns: accumulators (T per set), then ASTAGES x NS x 32 A columns.
    const uint32_t acc_col = 0;
    const uint32_t a_col0 = (uint32_t)(NS * T);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t stream_policy = ptx::policy_evict_first();
            ptx::prefetch_tmap(&tmap_a);
            ptx::prefetch_tmap(&tmap_w0);
            if (SWIGLU) ptx::prefetch_tmap(&tmap_w1);
            const uint32_t tx_bytes = (uint32_t)L.b_stage + (uint32_t)kChunk;
            int kb = 0, s = 0;
            uint32_t ph = 0;
            for (; kb < nkb; ++kb) {
                if (!ptx::mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.err, p.wait_ns)) break;
                // One box of COLS/16 sub-tiles x one k-block per weight set (sub-tiles
                // past N read as zero), full size in bytes whatever the ragged edge.
                ptx::mbar_arrive_expect_tx(&full[s], tx_bytes);
                ptx::tma_load_2d(smem + (size_t)s * L.b_stage, &tmap_a, kb * kKBlock, m0, &full[s]);
                unsigned char *wdst = smem + L.w_off + (size_t)s * kChunk;
                ptx::tma_load_3d_hint(wdst, &tmap_w0, 0, kb, sub0, &full[s], stream_policy);
                if (SWIGLU)  // up rows in the second half of the slot
                    ptx::tma_load_3d_hint(wdst + kChunk / 2, &tmap_w1, 0, kb, sub0, &full[s], stream_policy);
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (*abort_flag) {  // let issued copies land before the CTA can exit
                volatile int no_abort = 0;
                for (int s = 0; s < STAGES && s < kb; ++s) {
                    const int last = s + ((kb - 1 - s) / STAGES) * STAGES;
                    ptx::mbar_wait(&full[s], (uint32_t)(last / STAGES) & 1u, &no_abort, nullptr, 200000000ull);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // This one thread issues every MMA of the CTA and shares its scheduler with
        // three busy dequant warps, so its instructions per block weigh on the block
        // period: descriptors and tensor-memory addresses advance by constant steps
        // and the stage counters run without divisions.
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(T);
            // Start-address field of the descriptor in 16-byte units: +b_stage/16 per
            // stage, +2 per k16 step (32 bytes); shared addresses stay below 2^18, so
            // the 14-bit field never carries.
            const uint64_t bdesc0 = smem_desc_sw128(ptx::smem_u32(smem));
            const uint32_t bstage = (uint32_t)(L.b_stage >> 4);
            const uint32_t d_acc = tmem + acc_col, a_base0 = tmem + a_col0;
            int kb = 0, s = 0;  // stage of both rings
            uint32_t ph = 0;
            for (; kb < nkb; ++kb) {
                // The dequant group arrives on afull only after it has itself waited for
                // this stage's copies (weights and activations alike), so a completed
                // afull phase implies a completed full phase: no second wait here.
                if (!ptx::mbar_wait(&afull[s], ph, abort_flag, p.err, p.wait_ns)) break;
                tc_fence_after();
                const uint64_t bdesc = bdesc0 + (uint64_t)((uint32_t)s * bstage);
                const uint32_t a_base = a_base0 + (uint32_t)(s * NS * 32);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
#pragma unroll
                    for (int w = 0; w < NS; ++w)
                        tc_mma(d_acc + (uint32_t)(w * T), a_base + (uint32_t)(w * 32 + 8 * j), bdesc + 2u * j, idesc,
                               (kb > 0 || j > 0) ? 1u : 0u);
                }
                tc_commit(&empty[s]);  // frees the shared-memory and tensor-memory stages
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (kb == nkb) {
                tc_commit(accfull);
            } else {  // aborted: wait (bounded) for the MMAs already issued
                tc_commit(drain);
                volatile int no_abort = 0;
                ptx::mbar_wait(drain, 0u, &no_abort, nullptr, 200000000ull);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ dequant, then epilogue
        const int q = warp & 3;              // tensor-memory lane quarter of this warp
        const int hf = (warp - 2) >> 2;      // warp group: k-blocks kb = hf (mod kDqParts), epilogue column chunks
        const int r = q * 32 + lane;         // MMA row (= tensor-memory lane)
        // SwiGLU interleaves the sets by 16 rows: in each lane quarter, lanes 0-15 hold
        // the gate rows and lanes 16-31 the up rows of the same 16 output columns, so
        // the epilogue pairs them with one shuffle.
        const int wset = SWIGLU ? (r >> 4) & 1 : 0;
        const int rr = SWIGLU ? (r >> 5) * 16 + (r & 15) : r;  // output column within the CTA
        // The row's weight set, selected field by field (a run-time index into the
        // parameter array would copy it to the stack).
        const void *const w_scales = wset ? p.w[1].scales : p.w[0].scales;
        const uint8_t *const w_zp = wset ? p.w[1].zp : p.w[0].zp;
        const int n = n0 + rr;
        const bool row_ok = rr < R;
        const int sub = rr >> 4, g = r & 7, h = (r >> 3) & 1;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const int sh0 = 4 * h, sh1 = 4 * h + 8;  // nibble pairs (e0,e1) and (e2,e3) of this row
        constexpr int j0 = 0;                    // all k16 steps of the group's blocks
        uint32_t zz[NS][kSPW], ss[NS][kSPW];
        if (row_ok && hf < nkb) {
#pragma unroll
            for (int w = 0; w < NS; ++w) load_row_meta<GROUP>(p, w_scales, w_zp, n, hf, j0, zz[w], ss[w]);
        }
        bool aborted = false;
        for (int kb = hf; kb < nkb; kb += kDqParts) {
            const int s = kb % STAGES;  // stage of both rings
            const uint32_t ph = (uint32_t)(kb / STAGES) & 1u;
            if (!aborted && !ptx::mbar_wait(&full[s], ph, abort_flag, p.err, p.wait_ns)) aborted = true;
            if (!aborted && !ptx::mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.err, p.wait_ns)) aborted = true;
            if (aborted) break;
            // The group's next block's metadata, loaded early (it is used one block later).
            const int kbn = kb + kDqParts;
            uint32_t zzn[NS][kSPW], ssn[NS][kSPW];
            if (row_ok && kbn < nkb) {
                const bool same_group = (kbn * kKBlock) / GROUP == (kb * kKBlock) / GROUP;
#pragma unroll
                for (int w = 0; w < NS; ++w) {
                    if (same_group) {
#pragma unroll
                        for (int jj = 0; jj < kSPW; ++jj) {
                            zzn[w][jj] = zz[w][jj];
                            ssn[w][jj] = ss[w][jj];
                        }
                    } else {
                        load_row_meta<GROUP>(p, w_scales, w_zp, n, kbn, j0, zzn[w], ssn[w]);
                    }
                }
            }
#pragma unroll
            for (int w = 0; w < NS; ++w) {
                uint32_t col[8 * kSPW];
                if (row_ok) {
                    const unsigned char *chunk = smem + L.w_off + (size_t)(s * NS + w) * kChunk +
                                                 wset * (kChunk / 2) + sub * kSubBytes;
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        // The four words (k16 steps 0..3) of the row's lane slot for fragment column t.
                        const unsigned char *slotp = chunk + (4 * g + ((t + (g >> 1)) & 3)) * 16;
                        const uint4 v = *reinterpret_cast<const uint4 *>(slotp);
                        const uint32_t words[kSPW] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int jj = 0; jj < kSPW; ++jj) {
                            const uint32_t lo = ((words[jj] >> sh0) & 0x000F000Fu) | 0x64006400u;  // k +0/1
                            const uint32_t hi = ((words[jj] >> sh1) & 0x000F000Fu) | 0x64006400u;  // k +2/3
                            col[8 * jj + 2 * t] = hmul2(hsub2(lo, zz[w][jj]), ss[w][jj]);
                            col[8 * jj + 2 * t + 1] = hmul2(hsub2(hi, zz[w][jj]), ss[w][jj]);
                        }
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 8 * kSPW; ++c) col[c] = 0u;
                }
                const uint32_t ta = tmem + lane_base + a_col0 + (uint32_t)((s * NS + w) * 32);
                tmem_st_cols(ta, col);
            }
            tmem_wait_st();
            tc_fence_before();
            ptx::mbar_arrive(&afull[s]);
            if (kbn < nkb) {
#pragma unroll
                for (int w = 0; w < NS; ++w)
#pragma unroll
                    for (int jj = 0; jj < kSPW; ++jj) {
                        zz[w][jj] = zzn[w][jj];
                        ss[w][jj] = ssn[w][jj];
                    }
            }
        }
        // Epilogue: D[row r][token] -> Y[m0 + token][n]; the warps of a lane
        // quarter take alternate 16-column chunks.
        const bool acc_ok = !aborted && ptx::mbar_wait(accfull, 0u, abort_flag, p.err, p.wait_ns);
        if constexpr (!SWIGLU) {
            if (acc_ok) {
                tc_fence_after();
                for (int c0 = 16 * hf; c0 < T; c0 += 16 * kDqParts) {
                    uint32_t v[16];
                    tmem_ld16(tmem + lane_base + acc_col + (uint32_t)c0, v);
                    tmem_wait_ld();
                    if (row_ok) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int m = m0 + c0 + i;
                            if (m < p.M) p.Y[(size_t)m * p.N + n] = __float2half_rn(__uint_as_float(v[i]));
                        }
                    }
                }
            }
        } else {
            // Lane r holds the gate (lanes 0-15 of a quarter) or the up (16-31) row of
            // output column n: exchange half of each 16-token chunk with lane r ^ 16,
            // then the gate lane finishes tokens 0-7 and the up lane tokens 8-15.
            if (acc_ok) {
                tc_fence_after();
                const bool gate_lane = (lane & 16) == 0;
                for (int c0 = 16 * hf; c0 < T; c0 += 16 * kDqParts) {
                    uint32_t v[16];
                    tmem_ld16(tmem + lane_base + acc_col + (uint32_t)c0, v);
                    tmem_wait_ld();
                    const int mb = m0 + c0 + (gate_lane ? 0 : 8);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float own = __uint_as_float(gate_lane ? v[i] : v[8 + i]);
                        const float peer = __shfl_xor_sync(0xffffffffu, __uint_as_float(gate_lane ? v[8 + i] : v[i]), 16);
                        const float gv = gate_lane ? own : peer, uv = gate_lane ? peer : own;
                        const int m = mb + i;
                        if (row_ok && m < p.M) p.Y[(size_t)m * p.N + n] = __float2half_rn(silu_f32(gv) * uv);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side
template <int GROUP, bool SWIGLU>
cudaError_t launch_tc_one(const TcParams &p, int T, cudaStream_t s) {
    using Sh = TcShape;
    const int cols = SWIGLU ? 64 : kTileRows;  // output columns per CTA
    CUtensorMap map_a, map_w0, map_w1;
    if (!tmap_activations(&map_a, p.A, p.M, p.K, T)) return cudaErrorInvalidValue;
    if (!tmap_weights(&map_w0, p.w[0].q_rep, p.N, p.K, 1, cols / kSubRows)) return cudaErrorInvalidValue;
    if (!tmap_weights(&map_w1, p.w[1].q_rep, p.N, p.K, 1, cols / kSubRows)) return cudaErrorInvalidValue;
    const TcSmem L = tc_smem(T, Sh::STAGES, Sh::ASTAGES, Sh::NS);
    // One CTA per SM: the kernel takes all 512 tensor-memory columns.
    const size_t smem = (L.total + 1024 > 120 * 1024) ? L.total + 1024 : 120 * 1024;
    auto kern = tc_kernel<GROUP, SWIGLU>;
    cudaError_t e = ensure_max_dyn_smem(reinterpret_cast<const void *>(kern), 227 * 1024);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((p.M + T - 1) / T), (unsigned)((p.N + cols - 1) / cols), 1);
    kern<<<grid, kThreads, smem, s>>>(map_a, map_w0, map_w1, p, T);
    return cudaGetLastError();
}

template <bool SWIGLU>
cudaError_t launch_tc_group(const TcParams &p, int group, int T, cudaStream_t s) {
    switch (group) {
        case 16: return launch_tc_one<16, SWIGLU>(p, T, s);
        case 32: return launch_tc_one<32, SWIGLU>(p, T, s);
        case 64: return launch_tc_one<64, SWIGLU>(p, T, s);
        default: return launch_tc_one<128, SWIGLU>(p, T, s);
    }
}

}  // namespace

// Tokens per tile: the whole M rounded up to 16 when it fits, else the maximum.
int tc_tile_tokens(int M, bool swiglu) {
    (void)swiglu;  // both modes use the same tile
    const int tmax = TcShape::TMAX;
    const int t = (M + 15) / 16 * 16;
    return t < tmax ? t : tmax;
}

void tc_launch_shape(int M, int N, bool swiglu, int *ctas, int *threads, int *smem, int *stages) {
    using Sh = TcShape;
    const int T = tc_tile_tokens(M, swiglu);
    const int cols = swiglu ? 64 : kTileRows;
    const TcSmem L = tc_smem(T, Sh::STAGES, Sh::ASTAGES, Sh::NS);
    *ctas = ((M + T - 1) / T) * ((N + cols - 1) / cols);
    *threads = kThreads;
    *smem = (int)((L.total + 1024 > 120 * 1024) ? L.total + 1024 : 120 * 1024);
    *stages = Sh::STAGES;
}

cudaError_t launch_tc(const TcParams &p, int group, bool swiglu, cudaStream_t s) {
    const int T = tc_tile_tokens(p.M, swiglu);
    return swiglu ? launch_tc_group<true>(p, group, T, s) : launch_tc_group<false>(p, group, T, s);
}

}  // namespace w4a16
