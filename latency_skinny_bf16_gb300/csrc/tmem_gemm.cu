// tmem_gemm.cu -- the fifth-generation tensor-core backend: W and X boxes by
// tensor-map TMA, tcgen05.mma into tensor memory, the accumulator drained into
// fp32 registers after every ring stage.
//
// Design source: "GLM-5.2 Blackwell decode optimizations", section
// "Implementation breakdown" item 3 (the decode projections qkv_a / q_b /
// eh_proj: the skinny GEMM at small M and a separate GEMM at medium M, picked
// per (N, K) by measured speed) and item 2 (programmatic dependent launch),
// and "[Perf][Feat] Add generic cuteDSL LL BF16 router (GEMM)", item 2 (K split
// over the CTAs of a thread-block cluster, partial sums reduced through
// distributed shared memory).
//
// GB300 form.
//   * Work split.  W's rows are cut into groups of 8.  The grid has C row
//     ranges (clusters of S CTAs along K); range c holds the groups
//     [c*G/C, (c+1)*G/C), so no range has more than one group more than
//     another.  A range is walked as T tiles of at most VP rows (VP a multiple
//     of 8, at most 128); the MMA's M side is 64 or 128 rows, and rows past a
//     tile's last row are never stored.  The planner sizes the grid at two
//     CTAs per SM, so the next call's CTAs (programmatic dependent launch)
//     fill each SM as this call's CTAs leave it.
//   * Thread 0 drives the TMA engine (128-byte swizzle, rows past M or N and
//     columns past K read as zeros), every copy of a stage completing on its
//     "full" mbarrier.  When K is a multiple of 64 a stage is one copy of W
//     through a 3-D view [K/64][N][64] (box kb x VP rows, or VP - 8 for a
//     range's short last tile) and one of X (box kb x MT tokens); otherwise,
//     for each 64-element K box, the tile's rows as at most five boxes of
//     128 / 64 / 32 / 16 / 8 rows (one tensor map per height) and one box of
//     X.  W is a weight, so with PDL the W copies of the first ring pass go
//     out before griddepcontrol.wait.
//   * Thread 32 issues tcgen05.mma kind::f16 (bf16 x bf16 -> fp32; M = TM,
//     N = MT tokens, K = 16 each) into one of four sets of tensor-memory
//     accumulators in rotation, one set per chunk of ring stages holding at
//     most 16 MMAs.  A set holds P = 64 / MT accumulators of MT columns and
//     the chunk's MMAs go to them in turn (consecutive MMAs are independent,
//     so the tensor core pipelines them); each accumulator's first MMA of the
//     chunk overwrites, so no chain is longer than 16 MMAs, and the issuer
//     runs up to four chunks ahead of the draining warps.  tcgen05.commit
//     frees each ring stage and marks the set full at the end of its chunk.
//   * Warps 2..5 (one per lane quarter of tensor memory) wait for each
//     set, read its P accumulators with tcgen05.ld, add them in order into
//     fp32 registers (one
//     output row per thread, the tokens in registers) and release it.  The
//     tensor core's own accumulation is not round-to-nearest per add (its
//     error is biased; measured on same-sign data), so it is kept to one
//     chunk, and the chunk sums are added in order with rounded fp32 adds.
//   * S = 1: each tile's rows are stored once its last stage is drained.
//     S > 1 (one tile per CTA): after a cluster barrier every CTA sends the
//     rows owned by rank q into q's ring (slot = sending rank) with
//     st.shared::cluster; after a second barrier each owner adds slots
//     0..S-1 in that order.  Every order is fixed, so a plan's result is
//     bit-identical from run to run.
// Every mbarrier wait is bounded; a wait that gives up records an error in
// the device status word and the CTA winds down: copies in flight and issued
// MMAs are waited for (bounded), a CTA whose accumulator was not drained sends
// no partials, both cluster barriers are still passed, and tensor memory is
// freed only once every issued MMA is known to be complete.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tma.cuh"

namespace skinny {
namespace {

constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;
enum : int { kWaitAcc = 5, kWaitAccEmpty = 6 };
constexpr int kWMaps = 5;                      // W box heights 128, 64, 32, 16, 8 rows
constexpr int kAccWarp0 = 2;                   // warps 2..5 drain the accumulators

constexpr int kNAcc = 4;                       // accumulator sets in rotation, one per chunk
// Each set holds P = 64 / MT accumulators of MT columns: the MMAs of a chunk
// go to them in turn, so consecutive MMAs do not wait on each other's result
// (a dependent chain of small MMAs runs at the tensor core's latency, not its
// rate).  kNAcc x P x MT = 256 columns for every token bucket.
__host__ __device__ constexpr int tc_par(int MT) { return 64 / MT; }
__host__ __device__ constexpr int tmem_cols(int MT) { return kNAcc * tc_par(MT) * MT; }
// Ring stages per accumulator chunk: at most 16 MMAs (4 per 64-element box)
// accumulate in tensor memory before the chunk is drained into registers.
__host__ __device__ inline int tc_chunk_stages(int kb) { return kb >= 4 ? 1 : 4 / kb; }

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(slot), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

// Shared-memory matrix descriptor: K-major operand in 128-byte swizzle atoms
// (8 rows x 128 bytes, rows 128 bytes apart, atoms 1024 bytes apart; the
// leading-dimension offset is not used by this layout).  `saddr` is the
// atom-aligned tile base plus 32 bytes per 16-element K step.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: fp32 D, bf16 A and B, both K-major,
// N = MT (bits 17-22, N / 8), M = TM (bits 24-28, M / 16).
template <int MT, int TM>
__host__ __device__ constexpr uint32_t idesc_bf16() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(MT >> 3) << 17) | ((uint32_t)(TM >> 4) << 24);
}
// D[tmem] (+)= A[smem] . B[smem]^T; accumulate = 0 overwrites D.
__device__ __forceinline__ void umma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}
// Arrive on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar)
                 : "memory");
}
// 16 consecutive fp32 columns of this thread's lane (not yet waited for).
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
// Wait for this thread's tcgen05.ld; the registers are passed through the
// statement so no use of them can be scheduled above the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15])
                 :
                 : "memory");
}

struct TcMaps {
    CUtensorMap w[kWMaps];   // box heights 128, 64, 32, 16, 8 rows (64 K elements each)
    CUtensorMap x;           // box MT rows x 64 K elements
    // K % 64 == 0: a whole ring stage in one copy.  3-D views of W / X as
    // [K/64 boxes][rows][64 elements] (the box index strides 128 bytes), with
    // boxes of kb x (VP or VP - 8 rows) x 64 and kb x MT x 64; they land as
    // kb consecutive swizzled regions, the layout of a stage.
    CUtensorMap w3[2];
    CUtensorMap x3;
};

struct TcParams {
    void *Y;
    int64_t ldy;
    int M, N, K;
    int KS;          // K elements per cluster rank, a multiple of 64 * kb
    int kb;          // 64-element boxes per ring stage
    int stages;
    int G, C;        // 8-row groups of W, row ranges
    int vg;          // groups per tile (VP = 8 * vg rows)
    int *status;
    uint64_t budget_ns;
    int out_bf16;
    int stage3d;     // 1: K % 64 == 0, whole stages by the 3-D maps (tiles of VP or VP - 8 rows)
    int late;        // let the next launch start once the producer has issued every copy
    // fused query RMS norm (NORM instantiations only): X = xn = rms_norm(xr) * gamma
    const uint16_t *xr;
    int64_t ldxr;
    const uint16_t *gamma;
    float eps;
    uint16_t *xn;    // written by the CTAs of row range 0 (each its K slice)
    int64_t ldxn;
};

// Shared-memory layout from the 1024-byte aligned base: the ring (per stage:
// kb W regions of VP rows x 128 bytes, then kb X regions of MT rows x 128
// bytes, or no X regions when X is resident), the resident X (fused norm: nxb
// boxes of MT rows x 128 bytes, the rank's whole K slice), a pad the MMA may
// read past the last W region (rows VP..TM-1 of a tile are never stored), then
// the mbarriers, the tensor-memory address, two flags and the norm's scratch.
constexpr int kTcTailBytes = 16 + 4 * 16 + 4 * 4 * 16;
__host__ __device__ inline int tc_stage_bytes(int VP, int MT, int kb, int nxb) {
    return kb * (VP + (nxb ? 0 : MT)) * 128;
}
__host__ __device__ inline int tc_pad_bytes(int VP, int MT, int kb, int TM, int nxb) {
    const int over = (TM - VP) * 128 - (nxb ? nxb : kb) * MT * 128;
    return over > 0 ? over : 0;
}
__host__ __device__ inline int tc_layout_bytes(int VP, int MT, int kb, int stages, int TM, int nxb) {
    return stages * tc_stage_bytes(VP, MT, kb, nxb) + nxb * MT * 128 + tc_pad_bytes(VP, MT, kb, TM, nxb) +
           8 * (2 * stages + 2 * kNAcc + 3) + kTcTailBytes;
}

// The 3-D W map a tile of `rows` rows uses: 0 for VP rows, 1 for VP - 8, -1
// when whole-stage copies are off or the height is neither.
__host__ __device__ inline int tc_w3_map(int stage3d, int rows, int VP) {
    if (!stage3d) return -1;
    if (rows == VP) return 0;
    if (rows == VP - 8 && VP > 8) return 1;
    return -1;
}

__device__ __forceinline__ uint4 lds128(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)) : "memory");
    return v;
}
__device__ __forceinline__ void sts128(void *p, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" :: "r"(smem_u32(p)), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// 8 bf16 of a row starting at k0 (zeros past K), read through L2 (.cg: the
// row may have just been written by the preceding kernel).
__device__ __forceinline__ uint4 load_chunk_cg(const uint16_t *row, int k0, int K) {
    if ((reinterpret_cast<uintptr_t>(row + k0) & 15) == 0 && k0 + 8 <= K) return ldg_v4(row + k0);
    uint32_t w[4] = {0, 0, 0, 0};
    for (int e = 0; e < 8; ++e)
        if (k0 + e < K) w[e >> 1] |= (uint32_t)ldg_u16(row + k0 + e) << (16 * (e & 1));
    return make_uint4(w[0], w[1], w[2], w[3]);
}
// 8 bf16 gains from k0 (zeros past K), read-only path.
__device__ __forceinline__ uint4 load_gamma(const uint16_t *g, int k0, int K) {
    if ((reinterpret_cast<uintptr_t>(g + k0) & 15) == 0 && k0 + 8 <= K) return ldg_stream_v4(g + k0);
    uint32_t w[4] = {0, 0, 0, 0};
    for (int e = 0; e < 8; ++e)
        if (k0 + e < K) w[e >> 1] |= (uint32_t)ldg_stream_u16(g + k0 + e) << (16 * (e & 1));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Fused query RMS norm (one-rank plans: the resident X holds whole rows), run
// by the four draining warps (jt = 0..127, wq = warp 0..3 among them) once the
// raw rows have landed by TMA in the resident X, before any MMA: r_m =
// 1 / sqrtf(sum_k x^2 / K + eps) for every token, in the exact order of the
// standalone norm kernel (thread jt takes the 8-element chunks jt, jt + 128,
// ... of the row, one fused multiply-add per element, then a warp butterfly
// and the warps in order), so both give the same bits; then every element is
// replaced in place by bf16_rn((x * r_m) * g_k) in the swizzled layout the MMA
// reads.  Rows >= M and columns >= K hold zeros.  The CTAs of row range 0
// also store the normalised rows to xn.
template <int MT>
__device__ __forceinline__ void norm_prologue(const TcParams &p, uint8_t *xres, float *rstat, float *part,
                                              int nxb, bool write_xn, int jt, int wq, int lane) {
    const int K = p.K, M = p.M;
    const int chunks = (K + 7) / 8;
    float ss[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) ss[m] = 0.f;
    for (int c = jt; c < chunks; c += 128) {
        const int box = c >> 3, ch = c & 7;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                const uint4 q = lds128(xres + box * MT * 128 + m * 128 + ((ch ^ (m & 7)) << 4));
                const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float a = bf16_lo(w[e]), b = bf16_hi(w[e]);
                    ss[m] = fmaf(a, a, ss[m]);    // zeros past K add exactly nothing
                    ss[m] = fmaf(b, b, ss[m]);
                }
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss[m] += __shfl_xor_sync(0xFFFFFFFFu, ss[m], o);
    }
    if (lane == 0) {
#pragma unroll
        for (int m = 0; m < MT; ++m) part[wq * MT + m] = ss[m];
    }
    named_bar_sync(2, 128);
    if (jt < M) {
        float t = part[jt];
        for (int w = 1; w < 4; ++w) t += part[w * MT + jt];
        rstat[jt] = 1.0f / sqrtf(t / (float)K + p.eps);
    }
    named_bar_sync(2, 128);
    // one 8-element chunk per step, its gains loaded once for all tokens
    for (int cc = jt; cc < nxb * 8; cc += 128) {
        const int box = cc >> 3, ch = cc & 7;
        const int k0 = 8 * cc;
        const bool live = k0 < K;
        const uint4 gq = live ? load_gamma(p.gamma, k0, K) : make_uint4(0, 0, 0, 0);
        const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w};
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            uint8_t *addr = xres + box * MT * 128 + m * 128 + ((ch ^ (m & 7)) << 4);
            uint4 out = make_uint4(0, 0, 0, 0);
            if (m < M && live) {
                const uint4 raw = lds128(addr);
                const float r = rstat[m];
                const uint32_t xw[4] = {raw.x, raw.y, raw.z, raw.w};
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t lo = f32_to_bf16_rn(bf16_lo(xw[e]) * r * bf16_lo(gw[e]));
                    const uint32_t hi = f32_to_bf16_rn(bf16_hi(xw[e]) * r * bf16_hi(gw[e]));
                    o[e] = lo | (hi << 16);
                }
                out = make_uint4(o[0], o[1], o[2], o[3]);
                if (write_xn) {
                    uint16_t *dst = p.xn + (int64_t)m * p.ldxn + k0;
                    if ((reinterpret_cast<uintptr_t>(dst) & 15) == 0 && k0 + 8 <= K) {
                        *reinterpret_cast<uint4 *>(dst) = out;
                    } else {
                        for (int e = 0; e < 8 && k0 + e < K; ++e)
                            dst[e] = (uint16_t)(o[e >> 1] >> (16 * (e & 1)));
                    }
                }
            }
            sts128(addr, out);
        }
    }
    fence_proxy_async_smem();                    // generic-proxy writes, read next by the MMAs
    named_bar_sync(2, 128);
}

template <int MT, int TM, bool NORM>
__global__ void __launch_bounds__(kTcThreads, 2)
tmem_gemm_kernel(const __grid_constant__ TcMaps maps, const TcParams p)
{
    // the next call may start as soon as every CTA of this one is resident
    // (short calls), or once this CTA's producer has issued its last copy
    if (!p.late) griddep_launch_dependents();

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;            // 128-byte swizzle atoms: 1024-byte aligned
    uint8_t *smem = smem_raw + (base - raw);
    const int kb = p.kb, stages = p.stages;
    const int VP = 8 * p.vg;
    const int nxb = NORM ? p.KS / 64 : 0;                    // resident X boxes (fused norm)
    const int sbytes = tc_stage_bytes(VP, MT, kb, nxb);
    const uint32_t xres = base + stages * sbytes;
    const uint32_t bars = xres + nxb * MT * 128 + tc_pad_bytes(VP, MT, kb, TM, nxb);
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 8u * (stages + s); };
    auto accf = [&](int b) { return bars + 8u * (2 * stages + b); };
    auto acce = [&](int b) { return bars + 8u * (2 * stages + kNAcc + b); };
    const uint32_t done = bars + 8u * (2 * stages + 2 * kNAcc);
    const uint32_t xready = bars + 8u * (2 * stages + 2 * kNAcc + 1);   // fused norm: X is in place
    const uint32_t xraw = bars + 8u * (2 * stages + 2 * kNAcc + 2);     // fused norm: raw X has landed
    uint8_t *tail = smem + (bars - base) + 8 * (2 * stages + 2 * kNAcc + 3);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(tail);
    volatile int *fail = reinterpret_cast<volatile int *>(tail + 4);    // an accumulator was not drained
    volatile int *mma_ok = reinterpret_cast<volatile int *>(tail + 8);  // every issued MMA completed
    float *rstat = reinterpret_cast<float *>(tail + 16);               // fused norm: r per token
    float *npart = reinterpret_cast<float *>(tail + 16 + 4 * 16);      // fused norm: warp partial sums

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = gridDim.x;
    const int rank = (S > 1) ? (int)cluster_ctarank() : 0;
    // this CTA's rows [r0, r1) and K slice [kbeg, kend)
    const int c = blockIdx.y;
    const int g0 = (int)(((int64_t)c * p.G) / p.C), g1 = (int)(((int64_t)(c + 1) * p.G) / p.C);
    const int r0 = 8 * g0, r1 = 8 * g1;
    const int ntiles = (g1 - g0 + p.vg - 1) / p.vg;
    const int kbeg = rank * p.KS;
    const int kend = min(p.K, kbeg + p.KS);
    const int sk = 64 * kb;
    const int nk = kend > kbeg ? (kend - kbeg + sk - 1) / sk : 0;   // ring stages per tile
    const int total = ntiles * nk;
    const int cs = tc_chunk_stages(kb);                             // stages per accumulator chunk
    const int nchunk = (nk + cs - 1) / cs;                          // chunks per tile

    if (tid == 0) {
        for (int i = 0; i < kWMaps; ++i) prefetch_tensormap(&maps.w[i]);
        prefetch_tensormap(&maps.x);
        if (p.stage3d) {
            prefetch_tensormap(&maps.w3[0]);
            prefetch_tensormap(&maps.w3[1]);
            prefetch_tensormap(&maps.x3);
        }
        for (int s = 0; s < stages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < kNAcc; ++b) {
            mbar_init(accf(b), 1);
            mbar_init(acce(b), 4);            // lane 0 of each draining warp
        }
        mbar_init(done, 1);
        mbar_init(xready, 1);
        mbar_init(xraw, 1);
        *fail = 0;
        *mma_ok = 0;
        fence_mbarrier_init_cluster();
    }
    __syncthreads();

    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer
            auto tile_rows = [&](int t) { return min(VP, r1 - (r0 + t * VP)); };
            auto issue = [&](int i, int s, bool w_part, bool x_part) {
                const int t = i / nk, ks = i - t * nk;
                const int rows = tile_rows(t), row0 = r0 + t * VP;
                const uint32_t st = base + s * sbytes;
                const int w3 = tc_w3_map(p.stage3d, rows, VP);
                if (w3 >= 0 || (p.stage3d && !NORM)) {
                    const int kbox = (kbeg >> 6) + ks * kb;
                    if (w_part) {
                        if (w3 >= 0) {
                            tma_load_3d(st, &maps.w3[w3], row0, kbox, full(s));
                        } else {
                            // an odd tile height: per-box copies, regions VP rows apart
                            for (int b = 0; b < kb; ++b) {
                                int off = 0;
#pragma unroll
                                for (int h = 0; h < kWMaps; ++h) {
                                    const int height = 128 >> h;
                                    if (rows - off >= height) {
                                        tma_load_2d(st + b * VP * 128 + off * 128, &maps.w[h], kbeg + (ks * kb + b) * 64,
                                                    row0 + off, full(s));
                                        off += height;
                                    }
                                }
                            }
                        }
                    }
                    if (x_part && p.stage3d) tma_load_3d(st + kb * VP * 128, &maps.x3, 0, kbox, full(s));
                    else if (x_part)
                        for (int b = 0; b < kb; ++b)
                            tma_load_2d(st + kb * VP * 128 + b * MT * 128, &maps.x, kbeg + (ks * kb + b) * 64, 0, full(s));
                    return;
                }
                for (int b = 0; b < kb; ++b) {
                    const int k0 = kbeg + (ks * kb + b) * 64;
                    if (w_part) {
                        int off = 0;
#pragma unroll
                        for (int h = 0; h < kWMaps; ++h) {
                            const int height = 128 >> h;
                            if (rows - off >= height) {
                                tma_load_2d(st + b * VP * 128 + off * 128, &maps.w[h], k0, row0 + off, full(s));
                                off += height;
                            }
                        }
                    }
                    if (x_part) tma_load_2d(st + kb * VP * 128 + b * MT * 128, &maps.x, k0, 0, full(s));
                }
            };
            auto stage_tx = [&](int i) { return (uint32_t)(kb * (tile_rows(i / nk) + (NORM ? 0 : MT)) * 128); };
            const int pre = min(total, stages);
            for (int i = 0; i < pre; ++i) {
                mbar_arrive_expect_tx(full(i), stage_tx(i));
                issue(i, i, true, false);          // the weight: before the PDL wait
            }
            griddep_wait();
            if (!NORM)
                for (int i = 0; i < pre; ++i) issue(i, i, false, true);
            if (NORM) {
                // the raw rows of X (all K: the fused norm runs on one-rank plans), swizzled as the MMA reads them
                mbar_arrive_expect_tx(xraw, (uint32_t)(nxb * MT * 128));
                for (int b = 0; b < nxb; ++b) tma_load_2d(xres + b * MT * 128, &maps.x, b * 64, 0, xraw);
            }
            int issued = pre;
            for (int i = pre; i < total; ++i) {
                const int s = i % stages;
                if (!mbar_wait_bounded(empty(s), (uint32_t)((i / stages - 1) & 1), p.budget_ns)) {
                    report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitProducerEmpty);
                    break;
                }
                mbar_arrive_expect_tx(full(s), stage_tx(i));
                issue(i, s, true, !NORM);
                issued = i + 1;
            }
            if (p.late) griddep_launch_dependents();
            // every copy issued has landed before the ring is reused or the CTA exits
            for (int i = max(0, issued - stages); i < issued; ++i)
                if (!mbar_wait_bounded(full(i % stages), (uint32_t)((i / stages) & 1), kDrainNs))
                    report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitDrain);
        }
        __syncwarp();
    } else if (warp == 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), tmem_cols(MT));
        tc_fence_before();
        named_bar_sync(1, kTcThreads - 32);        // warps 1..5: the tensor-memory address is published
        tc_fence_after();
        const uint32_t tmem = *tmem_slot;
        if (lane == 0) {
            // ---- MMA issuer (its bounded waits start once the preceding kernel is done)
            griddep_wait();
            constexpr uint32_t idesc = idesc_bf16<MT, TM>();
            bool go = true;
            if (NORM && !mbar_wait_bounded(xready, 0, p.budget_ns)) {
                report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitX);
                go = false;
            }
            for (int i = 0; go && i < total; ++i) {
                const int s = i % stages;
                const int t = i / nk, ks = i - t * nk;
                const int g = t * nchunk + ks / cs;                 // accumulator chunk
                const int b = g % kNAcc;
                const bool first = (ks % cs) == 0, last = (ks % cs) == cs - 1 || ks == nk - 1;
                if (first && g >= kNAcc &&
                    !mbar_wait_bounded(acce(b), (uint32_t)((g / kNAcc - 1) & 1), p.budget_ns)) {
                    report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitAccEmpty);
                    break;
                }
                if (!mbar_wait_bounded(full(s), (uint32_t)((i / stages) & 1), p.budget_ns)) {
                    report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitConsumerFull);
                    break;
                }
                tc_fence_after();
                const uint32_t wst = base + s * sbytes;
                const uint32_t xst = NORM ? xres + ks * kb * MT * 128 : wst + kb * VP * 128;
                // a whole-stage 3-D copy packs the kb W regions at the tile's own height
                const int wrows = tc_w3_map(p.stage3d, min(VP, r1 - (r0 + t * VP)), VP) == 1 ? VP - 8 : VP;
                constexpr int P = tc_par(MT);
                const int q0 = (ks % cs) * 4 * kb;           // MMAs of this chunk issued so far
                for (int cb = 0; cb < kb; ++cb)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int q = q0 + 4 * cb + j;        // the chunk's first P MMAs overwrite
                        umma_bf16(tmem + (uint32_t)((b * P + q % P) * MT), sw128_desc(wst + cb * wrows * 128 + 32 * j),
                                  sw128_desc(xst + cb * MT * 128 + 32 * j), idesc, q < P ? 0u : 1u);
                    }
                umma_commit(empty(s));               // the stage is free once these MMAs have read it
                if (last) umma_commit(accf(b));      // the chunk's sum is complete
            }
            umma_commit(done);                       // tracks every MMA issued, also after a give-up
            if (mbar_wait_bounded(done, 0, kDrainNs)) *mma_ok = 1;
            else report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitDrain);
        }
        __syncwarp();
    } else {
        // ---- accumulator warps: lane quarter q of tensor memory
        named_bar_sync(1, kTcThreads - 32);
        tc_fence_after();
        const uint32_t tmem = *tmem_slot;
        griddep_wait();                          // Y may be read or written by the preceding kernel
        bool xok = true;
        if (NORM) {
            if (lane == 0) xok = mbar_wait_bounded(xraw, 0, p.budget_ns);
            xok = __shfl_sync(0xffffffffu, xok ? 1 : 0, 0) != 0;
            if (!xok && lane == 0) {
                report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitX);
                // the raw X copy is still in flight: let it land (bounded)
                // before the region is read, and before the CTA can exit
                if (!mbar_wait_bounded(xraw, 0, kDrainNs)) report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitDrain);
            }
            // every warp takes part in the barriers inside, whatever its wait gave
            norm_prologue<MT>(p, smem + (xres - base), rstat, npart, nxb, blockIdx.y == 0, tid - 64,
                              warp - kAccWarp0, lane);
        }
        if (NORM && tid == 64) mbar_arrive(xready);
        const int q = warp & 3;
        // accumulator row of this thread (M = 64: lanes 16..31 of each quarter hold none)
        const int row = (TM == 128) ? 32 * q + lane : 16 * q + lane;
        const bool has_row = (TM == 128) || lane < 16;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        const int M = p.M;
        float acc[MT];
#pragma unroll
        for (int j = 0; j < MT; ++j) acc[j] = 0.f;
        bool ok = true;
        for (int g = 0; g < ntiles * nchunk; ++g) {
            const int b = g % kNAcc;
            bool got = true;
            if (lane == 0) got = mbar_wait_bounded(accf(b), (uint32_t)((g / kNAcc) & 1), p.budget_ns);
            got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
            if (!got) {
                if (lane == 0) report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitAcc);
                ok = false;
                break;
            }
            tc_fence_after();
            // the chunk's P partial sums, added in a fixed order
            constexpr int P = tc_par(MT);
#pragma unroll
            for (int pp = 0; pp < P; ++pp) {
#pragma unroll
                for (int cc = 0; cc < MT / 16; ++cc) {
                    if (16 * cc < M) {            // warp-uniform
                        uint32_t r[16];
                        tmem_ld16_nowait(lane_base + (uint32_t)((b * P + pp) * MT + 16 * cc), r);
                        tmem_ld_wait(r);
#pragma unroll
                        for (int j = 0; j < 16; ++j) acc[16 * cc + j] += __uint_as_float(r[j]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce(b));
            if (S == 1 && (g % nchunk) == nchunk - 1) {
                // the tile's last chunk: store its rows
                const int t = g / nchunk;
                const int rows = min(VP, r1 - (r0 + t * VP));
                const int n = r0 + t * VP + row;
                if (has_row && row < rows && n < p.N) {
#pragma unroll
                    for (int m = 0; m < MT; ++m)
                        if (m < M) store_y(p.Y, p.out_bf16, m * p.ldy + n, acc[m]);
                }
#pragma unroll
                for (int j = 0; j < MT; ++j) acc[j] = 0.f;
            }
        }
        if (!ok) *fail = 1;
        // S > 1: one tile per CTA (the planner guarantees it); `acc` holds this
        // rank's partial sum (zeros for an empty K slice) until the reduction
        __syncthreads();                          // A: producer drained, MMAs complete
        if (S > 1) {
            cluster_arrive_release();             // B1: every CTA's ring is free
            cluster_wait_acquire();
            const int RQ = (VP + S - 1) / S;
            const int rows = min(VP, r1 - r0);
            if (has_row && row < rows && !*fail && *mma_ok) {
                const int qo = row / RQ, rl = row - qo * RQ;
                const uint32_t dst = mapa_shared(base, (uint32_t)qo);
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    if (m < M) st_shared_cluster_f32(dst + 4u * (uint32_t)((rank * M + m) * RQ + rl), acc[m]);
            }
            cluster_arrive_release();             // B2: every partial is in its owner's slots
            cluster_wait_acquire();
            const float *slots = reinterpret_cast<const float *>(smem);
            const int mine = max(0, min(RQ, rows - rank * RQ));
            for (int e = tid - kAccWarp0 * 32; e < M * mine; e += 4 * 32) {
                const int m = e / mine, r = e - m * mine;
                const int n = r0 + rank * RQ + r;
                float a = slots[m * RQ + r];
                for (int src = 1; src < S; ++src) a += slots[(src * M + m) * RQ + r];
                if (n < p.N) store_y(p.Y, p.out_bf16, m * p.ldy + n, a);
            }
        }
        tc_fence_before();
        __syncthreads();                          // C: tensor memory no longer read
        return;
    }

    // ---- producer and MMA warps: the same barriers as the draining warps
    __syncthreads();                              // A
    if (S > 1) {
        cluster_arrive_release();                 // B1
        cluster_wait_acquire();
        cluster_arrive_release();                 // B2
        cluster_wait_acquire();
    }
    __syncthreads();                              // C
    if (warp == 1) {
        tc_fence_after();
        if (*mma_ok) tmem_dealloc(*tmem_slot, tmem_cols(MT));
        // else: an issued MMA may still write this tensor memory; it stays
        // allocated until the CTA exits rather than being handed to another CTA
    }
}

using TcKernel = void (*)(const TcMaps, const TcParams);
const TcKernel kTc[3][2] = {{&tmem_gemm_kernel<16, 128, false>, &tmem_gemm_kernel<16, 64, false>},
                            {&tmem_gemm_kernel<32, 128, false>, &tmem_gemm_kernel<32, 64, false>},
                            {&tmem_gemm_kernel<64, 128, false>, &tmem_gemm_kernel<64, 64, false>}};
// the fused query RMS norm: up to 16 tokens
const TcKernel kTcNorm[2] = {&tmem_gemm_kernel<16, 128, true>, &tmem_gemm_kernel<16, 64, true>};

int tc_index(int M) { return M <= 16 ? 0 : M <= 32 ? 1 : 2; }

// Row split of a plan: groups per tile (vg) for C ranges of G groups, tiles
// of at most `max_vg` groups, as even as the ranges allow.
int tc_groups_per_tile(int G, int C, int max_vg) {
    const int gmax = (G + C - 1) / C;
    const int T = (gmax + max_vg - 1) / max_vg;
    return (gmax + T - 1) / T;
}

}  // namespace

// The driver's tensor-map encoder, resolved once through the runtime (no link
// against the driver library).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// bf16 [rows, cols] with row stride ld (elements), boxes of 64 columns x box_rows
// rows, 128-byte swizzle, zeros outside the tensor.
bool encode_bf16_2d(CUtensorMap *map, const void *ptr, int cols, int rows, int64_t ld, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 3-D view [ncols / 64][rows][64] of a bf16 [rows, ncols] matrix (ld in
// elements; ncols a multiple of 64), boxes of kb x box_rows x 64, 128-byte
// swizzle, zeros outside (box index or row past the end).
bool encode_bf16_3d(CUtensorMap *map, const void *ptr, int ncols, int rows, int64_t ld, int box_rows, int kb) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || ncols % 64) return false;
    const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(ncols / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)ld * 2, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)kb};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


int tc_tokens(int M) { return 16 << tc_index(M); }

bool tc_supported(int M) { return M >= 1 && M <= SKINNY_MAX_M; }

int tc_smem_bytes(int M, int N, int K, int block_n, int stage_k, int stages, int split_k, int clusters,
                  bool norm) {
    const int MT = tc_tokens(M);
    const int kb = stage_k / 64;
    const int G = (N + 7) / 8;
    const int vg = tc_groups_per_tile(G, clusters, block_n / 8);
    const int VP = 8 * vg;
    // fused norm: the rank's whole K slice of X stays in shared memory
    const int per_rank = ((K + stage_k - 1) / stage_k + split_k - 1) / split_k;
    const int nxb = norm ? per_rank * kb : 0;
    int bytes = tc_layout_bytes(VP, MT, kb, stages, block_n, nxb);
    // S > 1: the ring also receives the partials (S slots of M x ceil(VP / S) fp32)
    if (split_k > 1 && stages * tc_stage_bytes(VP, MT, kb, nxb) < split_k * M * ((VP + split_k - 1) / split_k) * 4)
        return 1 << 30;
    // cap the CTAs an SM can hold (two), so their tensor memory (256 columns
    // each) always fits in the SM's 512 columns
    const int min_smem = kTcMinSmem;
    if (bytes < min_smem - 1024) bytes = min_smem - 1024;
    return bytes + 1024;                         // slack for the 1024-byte alignment
}

// Default grid: a small cost model of what bounds the kernel, measured on GB300.
// Each candidate (cluster size S, row ranges C) is scored by its most loaded
// SM: the W bytes its CTAs stream (CTAs are placed evenly, so an SM holds
// ceil(CTAs / SMs) of them) over the smaller of the SM's share of HBM (about
// 45 GB/s) and the MMA issue rate (a small MMA about every 45 ns per SM,
// carrying 32 bytes of W per useful tile row).  Clustered grids are held to
// the clusters GB300 keeps resident at once (clusters of 4 and 8 do not fill
// every GPC) and pay about a microsecond for their reduction.  Every plan sizes
// its ring for two CTAs per SM: one CTA with a ring twice as deep streams
// slower (a CTA's copies land one stage at a time, about 0.85 us apart,
// whatever the depth).
namespace {
struct TcGrid { int S, C; double cost; };
TcGrid tc_default_grid(int G, int K, int bk, int num_sms, int force_s, int max_vg) {
    TcGrid best{0, 0, 1e30};
    const int nk_all = (K + bk - 1) / bk;
    const int slots = kTcCtasPerSm * num_sms;
    for (int S = 1; S <= kSplitMaxCluster; S *= 2) {
        if (force_s && S != force_s) continue;
        if (!force_s && S > 1 && nk_all < 2 * S) break;   // each rank keeps two stages of K
        // clusters resident at once at two CTAs per SM (cudaOccupancyMaxActiveClusters
        // on GB300): pairs fill every slot, fours and eights about 95%
        const int pct = S <= 2 ? 100 : 90;
        const int cap = (slots * pct) / (100 * S);
        int C = cap < G ? cap : G;
        if (S > 1 && (G + C - 1) / C > max_vg) continue;   // one tile per CTA
        if (C < 1) continue;
        const int gmax = (G + C - 1) / C;
        const int vg = tc_groups_per_tile(G, C, max_vg);
        const int ks = ((nk_all + S - 1) / S) * bk;
        const int kk = ks < K ? ks : K;
        const double cta_bytes = 8.0 * gmax * kk * 2.0;
        const int per_sm_ctas = (C * S + num_sms - 1) / num_sms;
        const double bw_hbm = 45e9, bw_mma = 32.0 * 8 * vg / 45e-9;
        const double cost = per_sm_ctas * cta_bytes / (bw_mma < bw_hbm ? bw_mma : bw_hbm) + (S > 1 ? 1e-6 : 0.0);
        if (cost < best.cost * 0.98) best = {S, C, cost};
    }
    return best;
}
}  // namespace

bool tc_make_plan(int M, int N, int K, int force_bn, int force_s, int force_stages, int force_bk, int force_c,
                  int num_sms, skinny_plan_t *p) {
    if (!tc_supported(M) || N < 1 || K < 1 || num_sms < 1) return false;
    if (force_bn && force_bn != 128 && force_bn != 64) return false;
    const int G = (N + 7) / 8;
    const int bk = force_bk ? force_bk : (K > 64 ? 128 : 64);
    if (bk < 64 || bk > kTcMaxBK || bk % 64) return false;
    const int nk_all = (K + bk - 1) / bk;         // ring stages over the whole K
    const int max_vg_default = (force_bn == 64) ? 8 : 16;
    int S = force_s, C = force_c;
    if (S == 0 || C == 0) {
        const TcGrid g = tc_default_grid(G, K, bk, num_sms, S, max_vg_default);
        if (g.S == 0) return false;
        if (S == 0) S = g.S;
        if (C == 0) C = g.C;
    }
    if (S < 1 || S > kSplitMaxCluster || (S & (S - 1))) return false;
    if (C < 1 || C > 65535 || C > G) return false;
    const int vg = tc_groups_per_tile(G, C, max_vg_default);
    const int VP = 8 * vg;
    if (S > 1 && (G + C - 1) / C > vg) return false;   // S > 1: one tile per CTA
    const int bn = force_bn ? force_bn : (VP <= 64 ? 64 : 128);
    if (VP > bn) return false;
    const int per_rank = (nk_all + S - 1) / S;    // ring stages per cluster rank (a forced S may leave
                                                  // the last ranks empty: they add zeros)
    const int ntiles_max = ((G + C - 1) / C + vg - 1) / vg;
    int stages = force_stages;
    if (!stages) {
        // two CTAs per SM: the ring within 110 KB
        stages = kSplitMaxStages;
        while (stages > 1 && tc_smem_bytes(M, N, K, bn, bk, stages, S, C, false) > kTcSmemBudget) --stages;
        // no deeper than the CTA's stages, but deep enough to receive the partials
        int least = 1;
        while (least < stages && tc_smem_bytes(M, N, K, bn, bk, least, S, C, false) > kMaxDynSmem) ++least;
        const int work = per_rank * ntiles_max;
        if (stages > work) stages = work > least ? work : least;
    }
    if (stages < 1 || stages > kSplitMaxStages) return false;
    const int smem = tc_smem_bytes(M, N, K, bn, bk, stages, S, C, false);
    if (smem > kMaxDynSmem) return false;
    p->backend = SKINNY_BACKEND_TCGEN05;
    p->consumer = SKINNY_CONSUMER_MMA;
    p->vec_elems = 8;
    p->block_n = bn;
    p->split_k = S;
    p->stages = stages;
    p->stage_k = bk;
    p->k_chunk = per_rank * bk;
    p->grid_x = S;
    p->grid_y = C;
    p->threads = kTcThreads;
    p->smem_bytes = smem;
    return true;
}

bool tc_make_norm_plan(int M, int N, int K, const skinny_plan_t &gemm, skinny_plan_t *p) {
    // one rank per range: the resident X then holds whole rows, so the raw rows
    // arrive by TMA once and the sum of squares reads them from shared memory
    if (gemm.backend != SKINNY_BACKEND_TCGEN05 || gemm.split_k != 1 || M < 1 || M > kTcNormMaxM) return false;
    *p = gemm;
    // the same split, tiles and stage length (so the same sums in the same
    // order) and the same CTAs per SM; the ring as deep as that budget leaves
    // beside the resident X (the whole SM only when the GEMM plan itself was
    // forced past two CTAs' budget)
    const int budget = gemm.smem_bytes > kTcSmemBudget + 2048 ? kMaxDynSmem : kTcSmemBudget;
    int stages = kSplitMaxStages;
    while (stages > 1 && tc_smem_bytes(M, N, K, gemm.block_n, gemm.stage_k, stages, gemm.split_k, gemm.grid_y,
                                       true) > budget)
        --stages;
    const int smem = tc_smem_bytes(M, N, K, gemm.block_n, gemm.stage_k, stages, gemm.split_k, gemm.grid_y, true);
    if (smem > kMaxDynSmem) return false;
    p->stages = stages;
    p->smem_bytes = smem;
    return true;
}

cudaError_t tc_prepare() {
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 2; ++j) {
            cudaError_t e = set_max_dyn_smem(kTc[i][j]);
            if (e != cudaSuccess) return e;
        }
    for (int j = 0; j < 2; ++j) {
        cudaError_t e = set_max_dyn_smem(kTcNorm[j]);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_tc(const GemmArgs &a, const skinny_plan_t &pl, const LaunchCtx &c, const TcNormArgs *norm) {
    const int S = pl.split_k;
    const int TM = pl.block_n;
    const int C = pl.grid_y;
    const int G = (a.N + 7) / 8;
    if (!tc_supported(a.M) || (TM != 128 && TM != 64) || S < 1 || S > kSplitMaxCluster || (S & (S - 1)) ||
        pl.stage_k < 64 || pl.stage_k > kTcMaxBK || pl.stage_k % 64 || pl.stages < 1 ||
        pl.stages > kSplitMaxStages || pl.k_chunk % pl.stage_k || (int64_t)pl.k_chunk * S < a.K || pl.grid_x != S ||
        C < 1 || C > G || C > 65535 || pl.threads != kTcThreads)
        return cudaErrorInvalidValue;
    const int vg = tc_groups_per_tile(G, C, TM / 8);
    if (8 * vg > TM || (S > 1 && (G + C - 1) / C > vg) ||
        pl.smem_bytes < tc_smem_bytes(a.M, a.N, a.K, TM, pl.stage_k, pl.stages, S, C, norm != nullptr) ||
        pl.smem_bytes > kMaxDynSmem)
        return cudaErrorInvalidValue;
    if (norm && (a.M > kTcNormMaxM || S != 1 || !norm->xr || !norm->gamma || !norm->xn || a.out_bf16))
        return cudaErrorInvalidValue;
    if ((reinterpret_cast<uintptr_t>(a.X) & 15) || (a.ldx & 7) || (reinterpret_cast<uintptr_t>(a.W) & 15) ||
        (a.ldw & 7))
        return cudaErrorInvalidValue;
    const int idx = tc_index(a.M);
    TcMaps maps;
    for (int h = 0; h < kWMaps; ++h)
        if (!encode_bf16_2d(&maps.w[h], a.W, a.K, a.N, a.ldw, 128 >> h)) return cudaErrorInvalidValue;
    // the fused norm's X map reads the raw rows; otherwise X itself
    if (norm && ((reinterpret_cast<uintptr_t>(norm->xr) & 15) || (norm->ldxr & 7))) return cudaErrorInvalidValue;
    if (!encode_bf16_2d(&maps.x, norm ? norm->xr : a.X, a.K, a.M, norm ? norm->ldxr : a.ldx, 16 << idx))
        return cudaErrorInvalidValue;
    // whole-stage copies when K is a whole number of 64-element boxes (a 3-D
    // view would otherwise read past the end of a row) and the maps encode
    const int VP = 8 * vg, kb = pl.stage_k / 64;
    int stage3d = (a.K % 64 == 0) ? 1 : 0;
    if (stage3d) {
        stage3d = encode_bf16_3d(&maps.w3[0], a.W, a.K, a.N, a.ldw, VP, kb) &&
                  encode_bf16_3d(&maps.w3[1], a.W, a.K, a.N, a.ldw, VP > 8 ? VP - 8 : 8, kb) &&
                  encode_bf16_3d(&maps.x3, norm ? norm->xr : a.X, a.K, a.M, norm ? norm->ldxr : a.ldx, 16 << idx, kb);
    }
    TcParams p;
    p.stage3d = stage3d;
    p.late = c.late ? 1 : 0;
    p.Y = a.Y;
    p.ldy = a.ldy;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.KS = pl.k_chunk;
    p.kb = pl.stage_k / 64;
    p.stages = pl.stages;
    p.G = G;
    p.C = C;
    p.vg = vg;
    p.status = c.status;
    p.budget_ns = c.budget_ns;
    p.out_bf16 = a.out_bf16;
    p.xr = norm ? norm->xr : nullptr;
    p.ldxr = norm ? norm->ldxr : 0;
    p.gamma = norm ? norm->gamma : nullptr;
    p.eps = norm ? norm->eps : 0.f;
    p.xn = norm ? norm->xn : nullptr;
    p.ldxn = norm ? norm->ldxn : 0;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, C, 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem_bytes;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = c.pdl ? 1 : 0;
    ++n;
    if (S > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = S;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, norm ? kTcNorm[TM == 128 ? 0 : 1] : kTc[idx][TM == 128 ? 0 : 1], maps, p);
}

}  // namespace skinny
