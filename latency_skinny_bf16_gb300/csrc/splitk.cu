// splitk.cu -- the cluster split-K backend of the skinny BF16 GEMM.
//
// Design source: "[Perf][Feat] Add generic cuteDSL LL BF16 router (GEMM)",
// section "Implementation breakdown" item 2 and the _ll_bf16_splitk.py
// snippet (K partitioned over the CTAs of a thread-block cluster; DMA producer
// warps and MMA consumer warps; a shared-memory pipeline of num_stages; the
// partial sums reduced across the cluster through distributed shared memory
// with st.shared::cluster), and the review notes on that page (the cluster
// barrier must be the non-.aligned form because the producer warp takes
// another branch).
//
// GB300 form.  The grid is S x C: clusters of S <= 8 CTAs along K, C clusters
// along N.  Each cluster loops over 16-row tiles of W (output columns)
// tile = y, y + C, ... (persistent when there are more tiles than clusters);
// CTA `rank` owns the K slice [rank*KS, rank*KS + KS) of every tile.
//   * Warp 4 is the producer: one lane per W row issues a 1-D bulk async copy
//     (cp.async.bulk, the TMA engine, no multicast) of the row's next BK = 256
//     elements into a `stages`-deep shared-memory ring, completing on the
//     stage's "full" mbarrier; it streams straight across tile boundaries.
//     W is a weight, so with PDL these copies are issued before
//     griddepcontrol.wait and overlap the preceding kernel.
//   * Warps 0-3 are consumers.  After griddepcontrol.wait they stage the CTA's
//     X slice in shared memory once, then for each ring stage either
//       FMA: warp w owns W rows 4w..4w+3, lane l the 8-element vector l of the
//            chunk; fp32 fused multiply-add into acc[M][4], or
//       MMA: mma.sync m16n8k16 with the 16 W rows on the MMA's M side and the
//            tokens on its N side (8, 16, 32 or 64 tokens: each A fragment
//            serves every 8-token group); ldmatrix feeds both
//            operands from padded (conflict-free) rows; the warps split the
//            chunk's 16-wide k steps, and each chunk's MMA sum is added into an
//            fp32 register accumulator with a plain rounded add,
//     and release the stage on its "empty" mbarrier.
//   * The per-CTA partial [M][16] of a tile goes to its owner CTA (column c
//     belongs to rank c % S) by st.shared::cluster into slot `rank` of the
//     tile's slot buffer (two buffers, alternating by tile); after one
//     barrier.cluster.arrive.release / wait.acquire every owner adds slots
//     0..S-1 in that order and writes Y, so the result is bit-identical from
//     run to run.  With S = 1 the partial is the result and goes to Y directly.
// Every mbarrier wait is bounded (see mbar_wait_bounded); a wait that gives
// up records an error in the device status word, waits (bounded) for its own
// copies in flight, and the CTA still takes part in every cluster barrier.
#include "common.cuh"
#include "internal.h"

namespace skinny {

namespace {

constexpr int kBN = 16;
// Ring rows hold `bk` K elements (bk a multiple of 64) plus 16 bytes of pad, so
// the row stride is 16 (mod 128) bytes and ldmatrix / 128-bit shared loads of
// 8 consecutive rows hit 8 different bank groups.
__host__ __device__ inline int ring_row_bytes(int bk) { return bk * 2 + 16; }
constexpr uint64_t kDrainBudgetNs = 200ull * 1000 * 1000;

struct Layout {
    int xrows, xrowb;
    int ring, xs, red, slots, bars, ctrl, total;
};

__host__ __device__ inline int round_up(int v, int a) { return (v + a - 1) / a * a; }

// Partial-sum slot buffers per CTA: two, alternating by tile, so persistent
// clusters can loop over tiles; one for 32 / 64 tokens, whose plans are never
// persistent (each cluster owns one tile), to keep shared memory in bounds.
__host__ __device__ constexpr int slot_buffers(int MT) { return MT >= 32 ? 1 : 2; }

// X holds the M real token rows only: the MMA consumer's fragment loads for
// tokens M..MT-1 (whose sums are dropped) read row 0 instead.
__host__ __device__ inline Layout make_layout(int MT, int M, int consumer, int stages, int KS, int S, int bk) {
    Layout L;
    (void)consumer;
    L.xrows = M;
    L.xrowb = round_up(KS * 2, 128) + 16;          // X row stride: 16 (mod 128)
    int off = 0;
    L.ring = off;  off += stages * kBN * ring_row_bytes(bk);
    L.xs = off;    off += L.xrows * L.xrowb;
    off = round_up(off, 16);
    L.red = off;   off += (consumer == SKINNY_CONSUMER_MMA) ? splitk_consumer_warps(consumer, MT, bk) * MT * kBN * 4 : 0;
    L.slots = off; off += (S > 1) ? slot_buffers(MT) * S * MT * kBN * 4 : 0;   // alternating by tile
    off = round_up(off, 8);
    L.bars = off;  off += 2 * stages * 8 + 8;      // full[stages], empty[stages], x_full
    L.ctrl = off;  off += 16;
    L.total = round_up(off, 128);
    return L;
}

struct SplitParams {
    const uint16_t *X; int64_t ldx;
    const uint16_t *W; int64_t ldw;
    void *Y; int64_t ldy;   // fp32, or bf16 bits when out_bf16
    int M, N, K;
    int KS;            // K elements per rank (multiple of 16)
    int bk;            // K elements per ring stage (multiple of 64, <= 2048)
    int stages;
    int x_vec16;       // X rows 16-byte aligned (vector staging)
    int *status;
    uint64_t budget_ns;
    int out_bf16;
    int late;          // let the next launch start once every W copy is issued
};

// Bounded wait used when draining: also stops early once the producer has
// given up before issuing the awaited chunk.
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, int g,
                                           volatile int *abort_flag, volatile int *issued) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag && *issued <= g) return false;   // never issued: nothing in flight
        if (globaltimer_ns() - t0 > kDrainBudgetNs) return false;
    }
}

template <int MT, int CONS, int CW>
__global__ void __launch_bounds__((CW + 1) * 32)
splitk_kernel(const SplitParams p)
{
    // CW consumer warps; warp CW produces
    extern __shared__ __align__(128) uint8_t smem[];
    const int S = gridDim.x;                       // CTAs per cluster along K
    const int C = gridDim.y;                       // clusters, persistent over row tiles
    const int T = (p.N + kBN - 1) / kBN;           // row tiles of 16
    const int my_tiles = ((int)blockIdx.y < T) ? (T - 1 - (int)blockIdx.y) / C + 1 : 0;
    const Layout L = make_layout(MT, p.M, CONS, p.stages, p.KS, S, p.bk);
    const int bk = p.bk;
    const int row_bytes = ring_row_bytes(bk);
    const int stage_bytes = kBN * row_bytes;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = (S > 1) ? (int)cluster_ctarank() : 0;
    const int kbeg = rank * p.KS;
    const int klen = max(0, min(p.K, kbeg + p.KS) - kbeg);
    const int nchunks = (klen + bk - 1) / bk;
    const int stages = p.stages;

    const uint32_t ring = smem_u32(smem + L.ring);
    const uint32_t full0 = smem_u32(smem + L.bars);
    const uint32_t empty0 = full0 + 8 * stages;
    const uint32_t xfull = empty0 + 8 * stages;
    // X slice by bulk copies when its rows are 16-byte aligned (klen % 8 == 0 always holds here)
    const bool bulk_x = p.x_vec16 && klen > 0 && my_tiles > 0;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.ctrl);
    volatile int *issued = abort_flag + 1;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, CW);
        }
        mbar_init(xfull, 1);
        *abort_flag = 0;
        *issued = 0;
        fence_mbarrier_init_cluster();
    }
    __syncthreads();
    // Cluster barrier phases (S > 1), each one split into arrive / wait and
    // executed by every thread of every CTA exactly once:
    //   phase 0      every CTA of the cluster has started (its shared memory
    //                may be written through DSMEM from then on);
    //   phase i + 1  every CTA has written its partials of tile i into the
    //                owners' slot buffer (i & 1) and has read its own slots of
    //                tile i - 1, so buffer (i + 1) & 1 is free again (32 / 64
    //                tokens: one buffer, and a cluster owns at most one tile).
    if (S > 1) cluster_arrive_relaxed();

    if (warp == CW) {
        // ============================ producer warp ============================
        // Streams (tile, chunk) pieces through the ring across tile boundaries.
        bool aborted = false;
        bool x_done = !bulk_x;
        // X is the preceding kernel's output: wait for it (PDL) only after the
        // first ring fill of W is in flight, then one bulk copy per X row.
        auto issue_x = [&]() {
            griddep_wait();
            if (lane == 0) mbar_arrive_expect_tx(xfull, (uint32_t)(p.M * klen * 2));
            __syncwarp();
            for (int r = lane; r < p.M; r += 32)
                bulk_copy_g2s(smem_u32(smem + L.xs) + r * L.xrowb, p.X + r * p.ldx + kbeg,
                              (uint32_t)(klen * 2), xfull);
            x_done = true;
        };
        int g = 0;
        for (int i = 0; i < my_tiles; ++i) {
            const int n0 = ((int)blockIdx.y + i * C) * kBN;
            const int rows = min(kBN, p.N - n0);
            const uint16_t *wbase = p.W + (int64_t)n0 * p.ldw + kbeg;
            for (int c = 0; c < nchunks; ++c, ++g) {
                if (!x_done && g == stages) issue_x();
                if (aborted) continue;
                const int s = g % stages;
                if (g >= stages) {
                    bool ok = true;
                    if (lane == 0) ok = mbar_wait_bounded(empty0 + 8 * s, ((g / stages) - 1) & 1, p.budget_ns);
                    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                    if (!ok) {
                        if (lane == 0) {
                            report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitProducerEmpty);
                            *abort_flag = 1;
                        }
                        aborted = true;
                        continue;
                    }
                }
                const int len = min(bk, klen - c * bk);
                const uint32_t full = full0 + 8 * s;
                if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)(rows * len * 2));
                __syncwarp();
                for (int r = lane; r < rows; r += 32)
                    bulk_copy_g2s(ring + s * stage_bytes + r * row_bytes,
                                  wbase + (int64_t)r * p.ldw + c * bk, (uint32_t)(len * 2), full);
                __syncwarp();
                if (lane == 0) *issued = g + 1;
            }
            // X must be in flight before the producer first waits on a cluster
            // phase: that phase needs the consumers, and they need X.
            if (!x_done) issue_x();
            if (i == 0 && !p.late) griddep_launch_dependents();
            if (S > 1) {
                cluster_wait();             // phase i
                cluster_arrive_relaxed();   // phase i + 1 (the producer writes no slots)
            }
        }
        if (!x_done) issue_x();
        if (my_tiles == 0 || p.late) griddep_launch_dependents();
        if (S > 1) cluster_wait();          // phase my_tiles
    } else {
        // ============================ consumer warps ============================
        griddep_wait();   // X may come from the preceding kernel; Y may still be read by it
        // ---- X[0:M, kbeg:kbeg+klen] in shared memory once (rows of L.xrowb bytes):
        // bulk copies from the producer, else staged here
        uint8_t *xs = smem + L.xs;
        if (bulk_x) {
            if (!mbar_wait_bounded(xfull, 0, p.budget_ns)) {
                if (lane == 0) report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitX);
                if (!mbar_wait_bounded(xfull, 0, kDrainBudgetNs) && lane == 0)
                    report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitDrain);
            }
        } else if (p.x_vec16) {
            const int nv = klen >> 3;
#pragma unroll 4
            for (int i = tid; i < p.M * nv; i += CW * 32) {
                const int m = i / nv, v = i - m * nv;
                *reinterpret_cast<uint4 *>(xs + m * L.xrowb + v * 16) =
                    ldg_v4(p.X + m * p.ldx + kbeg + 8 * v);
            }
        } else {
#pragma unroll 4
            for (int i = tid; i < p.M * klen; i += CW * 32) {
                const int m = i / klen, k = i - m * klen;
                *reinterpret_cast<uint16_t *>(xs + m * L.xrowb + 2 * k) = ldg_u16(p.X + m * p.ldx + kbeg + k);
            }
        }
        named_bar_sync(1, CW * 32);
        if (!p.late) griddep_launch_dependents();
        if (S > 1) cluster_wait();          // phase 0: every peer has started

        const uint32_t xs_u32 = smem_u32(xs);
        const uint32_t slots = smem_u32(smem + L.slots);
        float *red = reinterpret_cast<float *>(smem + L.red);   // MMA: [warp][MT][16]
        bool failed = false;
        int g = 0;
        for (int i = 0; i < my_tiles; ++i) {
            const int n0 = ((int)blockIdx.y + i * C) * kBN;
            const int rows = min(kBN, p.N - n0);
            const int sbuf = (slot_buffers(MT) == 2) ? (i & 1) : 0;
            const uint32_t slot_buf = slots + (uint32_t)(sbuf * S * MT * kBN * 4);

            constexpr int PM = (CONS == SKINNY_CONSUMER_FMA) ? MT : 1;
            constexpr int NT = (CONS == SKINNY_CONSUMER_MMA) ? MT / 8 : 1;   // n8 token tiles
            float part[PM][4];        // FMA: acc[m][r] for W rows 4*warp + r
#pragma unroll
            for (int m = 0; m < PM; ++m)
#pragma unroll
                for (int r = 0; r < 4; ++r) part[m][r] = 0.f;
            float macc[NT][4];        // MMA accumulators, one n8 token tile each
#pragma unroll
            for (int h = 0; h < NT; ++h)
#pragma unroll
                for (int q = 0; q < 4; ++q) macc[h][q] = 0.f;

            for (int c = 0; c < nchunks; ++c, ++g) {
                const int s = g % stages;
                const uint32_t full = full0 + 8 * s;
                const uint32_t par = (g / stages) & 1;
                if (!failed) {
                    if (*abort_flag && *issued <= g) {
                        failed = true;             // the producer gave up before this chunk
                    } else if (!mbar_wait_bounded(full, par, p.budget_ns)) {
                        failed = true;
                        if (lane == 0) report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitConsumerFull);
                        if (!drain_wait(full, par, g, abort_flag, issued) && lane == 0)
                            report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitDrain);
                    }
                } else if (!(*abort_flag && *issued <= g)) {
                    // already failed: still wait (bounded) for this chunk's copies
                    // so nothing lands in shared memory after the CTA exits
                    if (!drain_wait(full, par, g, abort_flag, issued) && lane == 0)
                        report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitDrain);
                }
                if (!failed) {
                    const int len = min(bk, klen - c * bk);
                    const uint32_t stage = ring + s * stage_bytes;
                    if constexpr (CONS == SKINNY_CONSUMER_FMA) {
                        const int nv = len >> 3;
                        const int r0 = warp * 4;
                        for (int j = lane; j < nv; j += 32) {
                            float w[4][8];
#pragma unroll
                            for (int r = 0; r < 4; ++r) {
                                uint4 v;
                                asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                             : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                                             : "r"(stage + (r0 + r) * row_bytes + j * 16));
                                w[r][0] = bf16_lo(v.x); w[r][1] = bf16_hi(v.x);
                                w[r][2] = bf16_lo(v.y); w[r][3] = bf16_hi(v.y);
                                w[r][4] = bf16_lo(v.z); w[r][5] = bf16_hi(v.z);
                                w[r][6] = bf16_lo(v.w); w[r][7] = bf16_hi(v.w);
                            }
                            const uint8_t *xcol = xs + (c * bk + j * 8) * 2;
#pragma unroll
                            for (int m = 0; m < MT; ++m) {
                                const uint4 v = *reinterpret_cast<const uint4 *>(xcol + m * L.xrowb);
                                float x[8];
                                x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
                                x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
#pragma unroll
                                for (int e = 0; e < 8; ++e)
#pragma unroll
                                    for (int r = 0; r < 4; ++r) part[m][r] = fmaf(x[e], w[r][e], part[m][r]);
                            }
                        }
                    } else {
                        // MMA: A = 16 W rows x 16 k (ldmatrix.x4), B = 16 k x MT tokens.
                        // The MMA sum is moved into the fp32 accumulator (a rounded
                        // add) after at most 4 k16 steps.  (Issuing every fragment load
                        // of the 4 steps first, into 4 independent MMA chains, measured
                        // no faster on GB300: the consumer is not what bounds this kernel.)
                        constexpr int GB = (MT <= 8) ? 1 : MT / 16;   // B fragments per step
                        const int steps = len >> 4;
                        const uint32_t a_row = (lane & 7) + 8 * ((lane >> 3) & 1);
                        const uint32_t a_addr0 = stage + a_row * row_bytes + (lane >> 4) * 16;
                        const uint32_t kh = (lane >> 3) & 1;
                        // byte offset of the X row this lane addresses in each B fragment
                        // (tokens past M read row 0; their sums are dropped)
                        uint32_t xrow[GB];
#pragma unroll
                        for (int h2 = 0; h2 < GB; ++h2) {
                            const int tok = (MT <= 8) ? (lane & 7) : (lane & 7) + 8 * (lane >> 4) + 16 * h2;
                            xrow[h2] = (uint32_t)((tok < p.M ? tok : 0) * L.xrowb);
                        }
                        for (int j0 = warp; j0 < steps; j0 += 4 * CW) {
                            float d[NT][4];
#pragma unroll
                            for (int h = 0; h < NT; ++h)
#pragma unroll
                                for (int q = 0; q < 4; ++q) d[h][q] = 0.f;
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const int j = j0 + q * CW;
                                if (j < steps) {
                                    uint32_t a[4];
                                    ldmatrix_x4(a_addr0 + j * 32, a[0], a[1], a[2], a[3]);
                                    const int kx = c * bk + j * 16;
                                    if constexpr (MT <= 8) {
                                        uint32_t b0, b1;
                                        ldmatrix_x2(xs_u32 + xrow[0] + (kx + 8 * kh) * 2, b0, b1);
                                        mma_bf16_16816(d[0], a, b0, b1, d[0]);
                                    } else {
                                        // 16 tokens per ldmatrix.x4; the A fragment serves every group
#pragma unroll
                                        for (int h2 = 0; h2 < GB; ++h2) {
                                            uint32_t b0, b1, b2, b3;
                                            ldmatrix_x4(xs_u32 + xrow[h2] + (kx + 8 * kh) * 2, b0, b1, b2, b3);
                                            mma_bf16_16816(d[2 * h2], a, b0, b1, d[2 * h2]);
                                            mma_bf16_16816(d[2 * h2 + 1], a, b2, b3, d[2 * h2 + 1]);
                                        }
                                    }
                                }
                            }
#pragma unroll
                            for (int h = 0; h < NT; ++h)
#pragma unroll
                                for (int q = 0; q < 4; ++q) macc[h][q] += d[h][q];
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8 * s);
            }

            // ---- the CTA's partial P[m][c] of this tile, to Y (S == 1) or to its owner
            auto emit = [&](int m, int c, float v) {
                if (m >= p.M || c >= rows) return;
                if (S == 1) {
                    store_y(p.Y, p.out_bf16, m * p.ldy + n0 + c, v);
                } else {
                    const uint32_t local = slot_buf + (uint32_t)(((rank * MT + m) * kBN + c) * 4);
                    st_shared_cluster_f32(mapa_shared(local, (uint32_t)(c % S)), v);
                }
            };
            if constexpr (CONS == SKINNY_CONSUMER_FMA) {
#pragma unroll
                for (int m = 0; m < MT; ++m)
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        float v = part[m][r];
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
                        part[m][r] = v;
                    }
                // every lane now holds all sums; lane l emits pairs l, l+32, ...
#pragma unroll
                for (int m = 0; m < MT; ++m)
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        if (((m * 4 + r) & 31) == lane) emit(m, warp * 4 + r, part[m][r]);
            } else {
                // fragment: thread (g4 = lane/4, t4 = lane%4) holds rows g4, g4+8
                // for tokens 2*t4, 2*t4+1 (+8 for the second MMA)
                const int g4 = lane >> 2, t4 = lane & 3;
#pragma unroll
                for (int h = 0; h < NT; ++h) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int tok = 8 * h + 2 * t4 + (q & 1);
                        const int row = g4 + 8 * (q >> 1);
                        if (tok < MT) red[(warp * MT + tok) * kBN + row] = macc[h][q];
                    }
                }
                named_bar_sync(1, CW * 32);
                for (int e = tid; e < MT * kBN; e += CW * 32) {
                    const int m = e / kBN, c = e - m * kBN;
                    float v = red[m * kBN + c];
#pragma unroll
                    for (int w = 1; w < CW; ++w) v += red[(w * MT + m) * kBN + c];
                    emit(m, c, v);
                }
                named_bar_sync(1, CW * 32);   // red is reused by the next tile
            }

            if (S > 1) {
                cluster_arrive_release();   // phase i + 1: partials of tile i are in the owners' slots
                cluster_wait_acquire();
                const float *sl = reinterpret_cast<const float *>(smem + L.slots) + sbuf * S * MT * kBN;
                for (int e = tid; e < MT * kBN; e += CW * 32) {
                    const int m = e / kBN, c = e - m * kBN;
                    if (m < p.M && c < rows && (c % S) == rank) {
                        float v = sl[(0 * MT + m) * kBN + c];
                        for (int r = 1; r < S; ++r) v += sl[(r * MT + m) * kBN + c];
                        store_y(p.Y, p.out_bf16, m * p.ldy + n0 + c, v);
                    }
                }
            }
        }
    }
}

using SplitKernel = void (*)(const SplitParams);

template <int MT> constexpr SplitKernel fma_k() { return &splitk_kernel<MT, SKINNY_CONSUMER_FMA, kSplitConsumerWarps>; }

const SplitKernel kFma[kMaxMSmall] = {
    fma_k<1>(), fma_k<2>(), fma_k<3>(), fma_k<4>(), fma_k<5>(), fma_k<6>(), fma_k<7>(), fma_k<8>(),
    fma_k<9>(), fma_k<10>(), fma_k<11>(), fma_k<12>(), fma_k<13>(), fma_k<14>(), fma_k<15>(), fma_k<16>()};
constexpr int kW4 = kSplitConsumerWarps, kW8 = kSplitMmaWarps;
const SplitKernel kMma[4] = {&splitk_kernel<8, SKINNY_CONSUMER_MMA, kW4>, &splitk_kernel<16, SKINNY_CONSUMER_MMA, kW4>,
                             &splitk_kernel<32, SKINNY_CONSUMER_MMA, kW4>, &splitk_kernel<64, SKINNY_CONSUMER_MMA, kW4>};
// stages of at least 1024 K elements, up to 16 tokens: 8 consumer warps
const SplitKernel kMma8[2] = {&splitk_kernel<8, SKINNY_CONSUMER_MMA, kW8>, &splitk_kernel<16, SKINNY_CONSUMER_MMA, kW8>};

int mma_index(int M) { return M <= 8 ? 0 : M <= 16 ? 1 : M <= 32 ? 2 : 3; }

}  // namespace

int splitk_mma_tokens(int M) { return M <= 8 ? 8 : M <= 16 ? 16 : M <= 32 ? 32 : 64; }

namespace {
int mt_for(int M, int consumer) { return consumer == SKINNY_CONSUMER_MMA ? splitk_mma_tokens(M) : M; }

}  // namespace

bool splitk_supported(int M, int consumer, int block_n) {
    return M >= 1 && block_n == kBN &&
           ((consumer == SKINNY_CONSUMER_FMA && M <= kMaxMSmall) ||
            (consumer == SKINNY_CONSUMER_MMA && M <= kMaxMSplitMma));
}

int splitk_smem_bytes(int M, int consumer, int block_n, int stages, int k_slice, int split_k, int bk) {
    (void)block_n;
    return make_layout(mt_for(M, consumer), M, consumer, stages, k_slice, split_k, bk).total;
}

cudaError_t splitk_prepare() {
    for (int m = 0; m < kMaxMSmall; ++m) {
        cudaError_t e = set_max_dyn_smem(kFma[m]);
        if (e != cudaSuccess) return e;
    }
    for (int i = 0; i < 4; ++i) {
        cudaError_t e = set_max_dyn_smem(kMma[i]);
        if (e != cudaSuccess) return e;
    }
    for (int i = 0; i < 2; ++i) {
        cudaError_t e = set_max_dyn_smem(kMma8[i]);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_splitk(const GemmArgs &a, const skinny_plan_t &pl, const LaunchCtx &c) {
    if (!splitk_supported(a.M, pl.consumer, pl.block_n)) return cudaErrorInvalidValue;
    if (pl.stage_k < 64 || pl.stage_k > kSplitMaxBK || pl.stage_k % 64) return cudaErrorInvalidValue;
    // a single slot buffer (32 / 64 tokens) is only safe when no cluster loops over tiles
    if (pl.split_k > 1 && pl.consumer == SKINNY_CONSUMER_MMA &&
        slot_buffers(splitk_mma_tokens(a.M)) == 1 && pl.grid_y < (a.N + kBN - 1) / kBN)
        return cudaErrorInvalidValue;
    SplitParams p;
    p.X = a.X; p.ldx = a.ldx; p.W = a.W; p.ldw = a.ldw; p.Y = a.Y; p.ldy = a.ldy;
    p.M = a.M; p.N = a.N; p.K = a.K;
    p.KS = pl.k_chunk;
    p.bk = pl.stage_k;
    p.stages = pl.stages;
    p.x_vec16 = ((reinterpret_cast<uintptr_t>(a.X) & 15) == 0 && (a.ldx & 7) == 0) ? 1 : 0;
    p.status = c.status;
    p.budget_ns = c.budget_ns;
    p.out_bf16 = a.out_bf16;
    p.late = c.late ? 1 : 0;
    const int cw = splitk_consumer_warps(pl.consumer, mt_for(a.M, pl.consumer), pl.stage_k);
    if (pl.threads != (cw + 1) * 32) return cudaErrorInvalidValue;
    SplitKernel fn = (pl.consumer != SKINNY_CONSUMER_MMA) ? kFma[a.M - 1]
                     : (cw == kSplitMmaWarps)            ? kMma8[mma_index(a.M)]
                                                         : kMma[mma_index(a.M)];

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.grid_x, pl.grid_y, 1);
    cfg.blockDim = dim3(pl.threads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem_bytes;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = c.pdl ? 1 : 0;
    ++n;
    if (pl.split_k > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = pl.split_k;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

}  // namespace skinny
