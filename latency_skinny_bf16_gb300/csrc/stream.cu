// stream.cu -- the K-outer streaming backend for large weights.
//
// Design source: the cluster split-K kernel of "[Perf][Feat] Add generic
// cuteDSL LL BF16 router (GEMM)", section "Implementation breakdown" item 2
// (a DMA producer warp feeding MMA consumer warps through a multi-stage
// shared-memory ring), applied to the large decode projections of "GLM-5.2
// Blackwell decode optimizations", Implementation breakdown item 3.
//
// GB300 form.  One CTA per SM (C CTAs, persistent): CTA b owns the 16-row
// tiles b, b + C, ... of W (at most kStreamMaxTiles of them) and the WHOLE K
// of each, so no partial sum ever leaves the CTA.  The loop order is K-outer:
// for every K chunk c of bk elements the ring receives, in this order,
//     X[0:M, chunk c]  then  W[tile i rows, chunk c] for each tile i,
// every row of each one bulk async copy (cp.async.bulk, the TMA engine).  The
// consumers keep the chunk's X entry while they run the chunk's W entries
// through mma.sync m16n8k16 (W rows on the MMA's M side, tokens on its N
// side), one register accumulator per tile, and release each entry on its
// "empty" mbarrier.  So X occupies one ring entry instead of a K slice (the
// cluster split-K kernel keeps M x K/S of X resident, which at large K leaves
// little room for W), and nothing synchronises the CTA between tiles: the
// producer streams W across tile and chunk boundaries, as deep as the ring.
// After the last chunk the four warps' sums of each tile are added in a fixed
// order in shared memory and written to Y, so results are bit-identical run
// to run.
//
// With PDL the first ring fill of W is issued before griddepcontrol.wait and
// the X entries right after it.  Every mbarrier wait is bounded; a wait that
// gives up records an error in the device status word and waits (bounded)
// for the copies already in flight before the CTA exits.
//
// Needs W rows and X rows 16-byte aligned (pointers and strides), K % 16 == 0,
// M <= 16, and a ring of at least (tiles per CTA + 1) entries.
#include "common.cuh"
#include "internal.h"

namespace skinny {
namespace {

constexpr int kBN = 16;
constexpr int kConsumerWarps = 4;
constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;

// Ring entries hold 16 rows of `bk` K elements plus 16 bytes of pad, so the
// row stride is 16 (mod 128) bytes: ldmatrix rows hit 8 different bank groups.
__host__ __device__ inline int entry_row_bytes(int bk) { return bk * 2 + 16; }

struct StreamLayout {
    int ring, red, bars, ctrl, total;
};

__host__ __device__ inline StreamLayout stream_layout(int MT, int stages, int bk) {
    StreamLayout L;
    int off = 0;
    L.ring = off;  off += stages * kBN * entry_row_bytes(bk);
    L.red = off;   off += kConsumerWarps * MT * kBN * 4;     // [warp][token][column]
    off = (off + 7) & ~7;
    L.bars = off;  off += 2 * stages * 8;                     // full[stages], empty[stages]
    L.ctrl = off;  off += 16;                                 // abort flag, entries issued
    L.total = (off + 127) & ~127;
    return L;
}

struct StreamParams {
    const uint16_t *X; int64_t ldx;
    const uint16_t *W; int64_t ldw;
    void *Y; int64_t ldy;   // fp32, or bf16 bits when out_bf16
    int M, N, K;
    int bk;                 // K elements per chunk (multiple of 64)
    int stages;             // ring entries, >= tiles per CTA + 1
    int *status;
    uint64_t budget_ns;
    int out_bf16;
    int late;               // let the next launch start once every W copy is issued
};

// Bounded wait while draining: stops early once the producer has given up
// before issuing the awaited entry (nothing of it is in flight then).
__device__ __forceinline__ bool drain_entry(uint32_t bar, uint32_t parity, int e, volatile int *abort_flag,
                                            volatile int *issued) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag && *issued <= e) return false;
        if (globaltimer_ns() - t0 > kDrainNs) return false;
    }
}

template <int MT>
__global__ void __launch_bounds__((kConsumerWarps + 1) * 32)
stream_kernel(const StreamParams p)
{
    constexpr int NT = MT / 8;   // n8 token tiles per MMA row block
    extern __shared__ __align__(128) uint8_t smem[];
    const int C = gridDim.x;
    const int T = (p.N + kBN - 1) / kBN;
    const int my_tiles = ((int)blockIdx.x < T) ? (T - 1 - (int)blockIdx.x) / C + 1 : 0;
    const int bk = p.bk, stages = p.stages;
    const int row_bytes = entry_row_bytes(bk);
    const int entry_bytes = kBN * row_bytes;
    const int nch = (p.K + bk - 1) / bk;
    const int per_chunk = my_tiles + 1;          // X entry, then one W entry per tile
    const int total = my_tiles > 0 ? nch * per_chunk : 0;
    const StreamLayout L = stream_layout(MT, stages, bk);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    const uint32_t ring = smem_u32(smem + L.ring);
    const uint32_t full0 = smem_u32(smem + L.bars);
    const uint32_t empty0 = full0 + 8 * stages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.ctrl);
    volatile int *issued = abort_flag + 1;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kConsumerWarps);
        }
        *abort_flag = 0;
        *issued = 0;
        fence_mbarrier_init_cluster();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ============================ producer warp ============================
        // entry e: chunk e / per_chunk; slot 0 of a chunk is X, slot i + 1 is tile i
        auto issue = [&](int e) {
            const int c = e / per_chunk, k = e - c * per_chunk;
            const int s = e % stages;
            const int len = min(bk, p.K - c * bk);
            const uint32_t full = full0 + 8 * s;
            const uint32_t dst = ring + s * entry_bytes;
            if (k == 0) {
                if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)(p.M * len * 2));
                __syncwarp();
                for (int r = lane; r < p.M; r += 32)
                    bulk_copy_g2s(dst + r * row_bytes, p.X + r * p.ldx + (int64_t)c * bk, (uint32_t)(len * 2), full);
            } else {
                const int n0 = ((int)blockIdx.x + (k - 1) * C) * kBN;
                const int rows = min(kBN, p.N - n0);
                if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)(rows * len * 2));
                __syncwarp();
                const uint16_t *wbase = p.W + (int64_t)n0 * p.ldw + (int64_t)c * bk;
                for (int r = lane; r < rows; r += 32)
                    bulk_copy_g2s(dst + r * row_bytes, wbase + (int64_t)r * p.ldw, (uint32_t)(len * 2), full);
            }
            __syncwarp();
        };
        const int fill = min(stages, total);
        // W is a weight: the first ring fill of W goes out before the wait for
        // the preceding kernel, whose output X may be
        for (int e = 0; e < fill; ++e)
            if (e % per_chunk != 0) issue(e);
        griddep_wait();
        for (int e = 0; e < fill; ++e)
            if (e % per_chunk == 0) issue(e);
        if (lane == 0) *issued = fill;
        if (!p.late) griddep_launch_dependents();
        for (int e = fill; e < total; ++e) {
            const int s = e % stages;
            bool ok = true;
            if (lane == 0) ok = mbar_wait_bounded(empty0 + 8 * s, ((e / stages) - 1) & 1, p.budget_ns);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitProducerEmpty);
                    *abort_flag = 1;
                }
                break;
            }
            issue(e);
            if (lane == 0) *issued = e + 1;
        }
        if (p.late) griddep_launch_dependents();
    } else {
        // ============================ consumer warps ============================
        griddep_wait();   // Y may still be read by the preceding kernel
        float acc[kStreamMaxTiles][NT][4];
#pragma unroll
        for (int i = 0; i < kStreamMaxTiles; ++i)
#pragma unroll
            for (int h = 0; h < NT; ++h)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[i][h][q] = 0.f;
        constexpr int GB = (MT <= 8) ? 1 : MT / 16;   // B fragments per k16 step
        const uint32_t a_off = ((lane & 7) + 8 * ((lane >> 3) & 1)) * row_bytes + (lane >> 4) * 16;
        const uint32_t kh = (lane >> 3) & 1;
        uint32_t xrow[GB];   // this lane's X row in each B fragment (tokens past M read row 0)
#pragma unroll
        for (int h2 = 0; h2 < GB; ++h2) {
            const int tok = (MT <= 8) ? (lane & 7) : (lane & 7) + 8 * (lane >> 4) + 16 * h2;
            xrow[h2] = (uint32_t)((tok < p.M ? tok : 0) * row_bytes) + kh * 16;
        }
        bool failed = false;
        // wait for entry e; after a failure keep waiting (bounded) for what is
        // in flight so nothing lands in shared memory after the CTA exits
        auto wait_entry = [&](int e) -> bool {
            const uint32_t bar = full0 + 8 * (e % stages);
            const uint32_t par = (e / stages) & 1;
            if (!failed) {
                if (*abort_flag && *issued <= e) {
                    failed = true;
                } else if (!mbar_wait_bounded(bar, par, p.budget_ns)) {
                    failed = true;
                    if (lane == 0) report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitConsumerFull);
                    if (!drain_entry(bar, par, e, abort_flag, issued) && lane == 0)
                        report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitDrain);
                }
                return !failed;
            }
            if (!(*abort_flag && *issued <= e) && !drain_entry(bar, par, e, abort_flag, issued) && lane == 0)
                report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitDrain);
            return false;
        };
        auto release = [&](int e) {
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * (e % stages));
        };
        for (int c = 0; c < nch && my_tiles > 0; ++c) {
            const int e0 = c * per_chunk;
            const bool have_x = wait_entry(e0);
            const uint32_t xs = ring + (e0 % stages) * entry_bytes;
            const int steps = min(bk, p.K - c * bk) >> 4;
#pragma unroll
            for (int i = 0; i < kStreamMaxTiles; ++i) {
                if (i < my_tiles) {
                    const int e = e0 + 1 + i;
                    if (wait_entry(e) && have_x) {
                        const uint32_t ws = ring + (e % stages) * entry_bytes + a_off;
                        // the 4 warps split the chunk's k16 steps; each MMA sum of up
                        // to 4 steps is added into the fp32 accumulator (rounded add)
                        for (int j0 = warp; j0 < steps; j0 += 4 * kConsumerWarps) {
                            float d[NT][4];
#pragma unroll
                            for (int h = 0; h < NT; ++h)
#pragma unroll
                                for (int q = 0; q < 4; ++q) d[h][q] = 0.f;
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const int j = j0 + q * kConsumerWarps;
                                if (j < steps) {
                                    uint32_t a[4];
                                    ldmatrix_x4(ws + j * 32, a[0], a[1], a[2], a[3]);
                                    if constexpr (MT <= 8) {
                                        uint32_t b0, b1;
                                        ldmatrix_x2(xs + xrow[0] + j * 32, b0, b1);
                                        mma_bf16_16816(d[0], a, b0, b1, d[0]);
                                    } else {
#pragma unroll
                                        for (int h2 = 0; h2 < GB; ++h2) {
                                            uint32_t b0, b1, b2, b3;
                                            ldmatrix_x4(xs + xrow[h2] + j * 32, b0, b1, b2, b3);
                                            mma_bf16_16816(d[2 * h2], a, b0, b1, d[2 * h2]);
                                            mma_bf16_16816(d[2 * h2 + 1], a, b2, b3, d[2 * h2 + 1]);
                                        }
                                    }
                                }
                            }
#pragma unroll
                            for (int h = 0; h < NT; ++h)
#pragma unroll
                                for (int q = 0; q < 4; ++q) acc[i][h][q] += d[h][q];
                        }
                    }
                    release(e);
                }
            }
            release(e0);
        }

        // ---- per tile: the 4 warps' sums added in warp order, then Y
        float *red = reinterpret_cast<float *>(smem + L.red);
        const int g4 = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int i = 0; i < kStreamMaxTiles; ++i) {
            if (i < my_tiles) {
                const int n0 = ((int)blockIdx.x + i * C) * kBN;
                const int rows = min(kBN, p.N - n0);
#pragma unroll
                for (int h = 0; h < NT; ++h)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int tok = 8 * h + 2 * t4 + (q & 1);
                        const int row = g4 + 8 * (q >> 1);
                        red[(warp * MT + tok) * kBN + row] = acc[i][h][q];
                    }
                named_bar_sync(1, kConsumerWarps * 32);
                for (int e = tid; e < MT * kBN; e += kConsumerWarps * 32) {
                    const int m = e / kBN, col = e - m * kBN;
                    if (m < p.M && col < rows) {
                        float v = red[m * kBN + col];
#pragma unroll
                        for (int w = 1; w < kConsumerWarps; ++w) v += red[(w * MT + m) * kBN + col];
                        store_y(p.Y, p.out_bf16, m * p.ldy + n0 + col, v);
                    }
                }
                named_bar_sync(1, kConsumerWarps * 32);   // red is reused by the next tile
            }
        }
    }
}

using StreamKernel = void (*)(const StreamParams);
const StreamKernel kStream[2] = {&stream_kernel<8>, &stream_kernel<16>};

}  // namespace

bool stream_supported(int M) { return M >= 1 && M <= kMaxMSmall; }

int stream_smem_bytes(int M, int stages, int bk) {
    return stream_layout(M <= 8 ? 8 : 16, stages, bk).total;
}

cudaError_t stream_prepare() {
    for (int i = 0; i < 2; ++i) {
        cudaError_t e = set_max_dyn_smem(kStream[i]);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_stream(const GemmArgs &a, const skinny_plan_t &pl, const LaunchCtx &c) {
    if (!stream_supported(a.M) || a.K % 16 != 0) return cudaErrorInvalidValue;
    if (pl.stage_k < 64 || pl.stage_k > kSplitMaxBK || pl.stage_k % 64) return cudaErrorInvalidValue;
    const int T = (a.N + kBN - 1) / kBN;
    const int per_cta = (T + pl.grid_x - 1) / pl.grid_x;
    // the ring must hold one chunk's X entry and every W entry of it, plus one
    if (per_cta > kStreamMaxTiles || pl.stages < per_cta + 1 || pl.stages > kSplitMaxStages)
        return cudaErrorInvalidValue;
    StreamParams p;
    p.X = a.X; p.ldx = a.ldx; p.W = a.W; p.ldw = a.ldw; p.Y = a.Y; p.ldy = a.ldy;
    p.M = a.M; p.N = a.N; p.K = a.K;
    p.bk = pl.stage_k;
    p.stages = pl.stages;
    p.status = c.status;
    p.budget_ns = c.budget_ns;
    p.out_bf16 = a.out_bf16;
    p.late = c.late ? 1 : 0;
    StreamKernel fn = kStream[a.M <= 8 ? 0 : 1];

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.grid_x, 1, 1);
    cfg.blockDim = dim3((kConsumerWarps + 1) * 32, 1, 1);
    cfg.dynamicSmemBytes = pl.smem_bytes;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = c.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

}  // namespace skinny
