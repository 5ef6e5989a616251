// dotmma.cu -- the dot-product backend with tensor-core arithmetic.
//
// Same division of work as the dot-product kernel ("[Perf][Feat] Add generic
// cuteDSL LL BF16 router (GEMM)", Implementation breakdown item 1: a CTA owns
// a block of output columns and the whole K, W streamed with 128-bit loads,
// partial sums reduced inside the CTA), with the multiply-adds done by
// mma.sync m16n8k16 (bf16 -> fp32) instead of CUDA-core FMA: at M >= 4 the
// FMA count per W element, not HBM, limits the FMA kernel.
//
// GB300 form.  A CTA of 4 warps owns RT tiles of 16 W rows (16*RT output
// columns).  Warp w works on tile w % RT and on every P-th 32-element K step
// (P = 4 / RT parts, interleaved so that the CTA's loads of a row are
// contiguous).  For one 32-element step of its tile, lane (g = lane/4,
// t = lane%4) loads W[row g][8t .. 8t+7] and W[row g+8][8t .. 8t+7] straight
// from HBM into registers (two 128-bit non-allocating loads), and X[token][8t ..
// 8t+7] from shared memory.  Those eight K values feed two m16n8k16 MMAs: the
// MMA's k slots {2t, 2t+1} take physical k = 8t + {0,1} (first MMA) or
// 8t + {4,5} (second), slots {2t+8, 2t+9} take 8t + {2,3} or 8t + {6,7}.  The
// same mapping is applied to A (W) and B (X), so each MMA still sums matching
// products; the 16 rows of W sit on the MMA's M side and the tokens on its N
// side (8 or 16 tokens).  Batches of 4 steps are double-buffered in registers
// (triple-buffered at 16 tokens: measured 31.3 -> 17.5 us on 24576 x 1536);
// each batch's MMA sum is added into an fp32 register accumulator with a plain
// rounded add.  The parts of a tile are added in a fixed order in shared
// memory, so a plan's result is bit-identical from run to run.
//
// Cluster split of K (up to 16 tokens).  On small weights (the router shapes)
// the CTAs of one column block are too few to keep HBM busy, so K is cut
// into S slices of KS elements (a multiple of 32) taken by the S CTAs of a
// thread-block cluster (grid S x blocks).  Each CTA sums its slice as above;
// its partial of output (column c of the block, token m) goes by
// st.shared::cluster into slot `rank` of CTA c % S, and after one
// barrier.cluster arrive.release / wait.acquire that owner adds slots
// 0..S-1 in order and writes Y: still bit-identical from run to run.  W
// moves by plain 128-bit loads, every one of a CTA's loads in flight at once,
// so a slice costs one DRAM round trip however short it is (the bulk-copy
// ring of the split-K backend pays an issue cost per W row and stage).
//
// X sits in shared memory with a row stride of 64 (mod 128) bytes, so the
// 128-bit reads of a quarter-warp (two rows x four 16-byte pieces) hit eight
// different bank groups.  X rows that are 16-byte aligned arrive by bulk async
// copies (one per row) on a bounded mbarrier wait, else by ordinary loads; X
// longer than the shared-memory budget is staged in chunks.  With PDL the
// first batch of W loads is issued before griddepcontrol.wait.
//
// Needs W rows 16-byte aligned (W and ldw) and K % 32 == 0.
#include "common.cuh"
#include "internal.h"

namespace skinny {
namespace {

constexpr int kWarps = kDotThreads / 32;
constexpr int kU = 4;   // 32-element K steps per warp per batch

__host__ __device__ inline int xrow_bytes(int kc) { return ((kc * 2 + 127) & ~127) + 64; }

}  // namespace

// K elements per cluster rank: ceil(K / S) rounded up to a whole 32-element step.
__host__ __device__ int dotmma_k_slice(int K, int S) { return ((K + S - 1) / S + 31) / 32 * 32; }

// A split is usable when every rank gets some K and the partial slots stay small
// (up to 16 tokens, clusters of up to 8).
bool dotmma_split_ok(int M, int K, int S) {
    if (S == 1) return true;
    if (S < 1 || S > kSplitMaxCluster || M > 16) return false;
    return (int64_t)(S - 1) * dotmma_k_slice(K, S) < K;
}

namespace {

__device__ __forceinline__ uint4 lds128(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }

template <int MT, int RT>
__global__ void __launch_bounds__(kDotThreads)
dotmma_kernel(const uint16_t *__restrict__ X, int64_t ldx,
              const uint16_t *__restrict__ W, int64_t ldw,
              void *__restrict__ Y, int64_t ldy,
              int M, int N, int K, int kc, int x_vec16, int *status, uint64_t budget_ns, int out_bf16, int S,
              int late)
{
    constexpr int P = kWarps / RT;    // K parts per row tile
    constexpr int NT = MT / 8;        // n8 token tiles
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t xbar_storage;
    const int xrowb = xrow_bytes(kc);
    uint8_t *xs = smem;                                              // [MT][xrowb]
    float *red = reinterpret_cast<float *>(smem + MT * xrowb);       // [RT][P][16][MT]
    float *slots = red + kWarps * 16 * MT;                           // S > 1: [S][RT * 16][MT]

    // S > 1: grid S x blocks, this CTA takes K slice `rank` of column block `blk`
    const int rank = (S > 1) ? (int)blockIdx.x : 0;
    const int blk = (S > 1) ? (int)blockIdx.y : (int)blockIdx.x;
    const int KS = (S > 1) ? dotmma_k_slice(K, S) : K;
    const int kbeg = rank * KS, kend = min(K, kbeg + KS);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tile = warp % RT, part = warp / RT;
    const int g = lane >> 2, t = lane & 3;
    const int n0 = (blk * RT + tile) * 16;
    // rows past N re-read row N-1; their sums are dropped
    const uint16_t *w0 = W + (int64_t)min(n0 + g, N - 1) * ldw + 8 * t;
    const uint16_t *w1 = W + (int64_t)min(n0 + g + 8, N - 1) * ldw + 8 * t;
    const uint32_t xbar = smem_u32(&xbar_storage);
    if (tid == 0) {
        mbar_init(xbar, 1);
        fence_mbarrier_init_cluster();
    }
    __syncthreads();
    if (S > 1) cluster_arrive_relaxed();   // phase 0: this CTA's slots may be written from now on

    float macc[NT][4];
#pragma unroll
    for (int h = 0; h < NT; ++h)
#pragma unroll
        for (int q = 0; q < 4; ++q) macc[h][q] = 0.f;

    // Batches of W in registers: 2 (one in flight while one is consumed), or 3
    // at 16 tokens, whose batches take twice the MMAs and shared-memory reads
    constexpr int NB = (MT == 16) ? 3 : 2;
    uint4 A0[NB][kU], A1[NB][kU];
    // batch starting at local step index j0: steps s = part + P * (j0 + u)
    auto load = [&](uint4 (&a0)[kU], uint4 (&a1)[kU], int k0, int nsteps, int j0) {
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int s = part + P * (j0 + u);
            if (s < nsteps) {
                a0[u] = ldg_stream_v4(w0 + k0 + s * 32);
                a1[u] = ldg_stream_v4(w1 + k0 + s * 32);
            }
        }
    };
    auto compute = [&](const uint4 (&a0)[kU], const uint4 (&a1)[kU], int nsteps, int j0) {
        float d[NT][4];
#pragma unroll
        for (int h = 0; h < NT; ++h)
#pragma unroll
            for (int q = 0; q < 4; ++q) d[h][q] = 0.f;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int s = part + P * (j0 + u);
            if (s < nsteps) {
                const uint8_t *xp = xs + g * xrowb + (s * 32 + 8 * t) * 2;
                uint4 xv[NT];
#pragma unroll
                for (int h = 0; h < NT; ++h) xv[h] = lds128(xp + h * 8 * xrowb);
                const uint32_t fa[4] = {a0[u].x, a1[u].x, a0[u].y, a1[u].y};   // k = 8t + 0..3
                const uint32_t fb[4] = {a0[u].z, a1[u].z, a0[u].w, a1[u].w};   // k = 8t + 4..7
#pragma unroll
                for (int h = 0; h < NT; ++h) {
                    mma_bf16_16816(d[h], fa, xv[h].x, xv[h].y, d[h]);
                    mma_bf16_16816(d[h], fb, xv[h].z, xv[h].w, d[h]);
                }
            }
        }
#pragma unroll
        for (int h = 0; h < NT; ++h)
#pragma unroll
            for (int q = 0; q < 4; ++q) macc[h][q] += d[h][q];
    };

    load(A0[0], A1[0], kbeg, max(0, min(kc, kend - kbeg)) / 32, 0);   // W is a weight: in flight before the PDL wait
    if constexpr (NB == 3) load(A0[1], A1[1], kbeg, max(0, min(kc, kend - kbeg)) / 32, kU);
    griddep_wait();
    if (!late) griddep_launch_dependents();

    for (int k0 = kbeg; k0 < kend; k0 += kc) {
        const int klen = min(kc, kend - k0);
        const int nsteps = klen / 32;
        if (k0 > kbeg) {
            __syncthreads();                     // every warp is done with the previous X chunk
            load(A0[0], A1[0], k0, nsteps, 0);
            if constexpr (NB == 3) load(A0[1], A1[1], k0, nsteps, kU);
        }
        // ---- stage X[0:M, k0:k0+klen] (klen is a multiple of 32)
        if (x_vec16) {
            if (warp == 0) {
                if (lane == 0) {
                    fence_proxy_async_smem();
                    mbar_arrive_expect_tx(xbar, (uint32_t)(M * klen * 2));
                }
                __syncwarp();
                for (int r = lane; r < M; r += 32)
                    bulk_copy_g2s(smem_u32(xs + r * xrowb), X + r * ldx + k0, (uint32_t)(klen * 2), xbar);
            }
            const uint32_t par = (uint32_t)(((k0 - kbeg) / kc) & 1);
            if (!mbar_wait_bounded(xbar, par, budget_ns)) {
                if (lane == 0) report_status(status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitX);
                if (!mbar_wait_bounded(xbar, par, 200ull * 1000 * 1000) && lane == 0)
                    report_status(status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitDrain);
            }
        } else {
#pragma unroll 4
            for (int i = tid; i < M * klen; i += kDotThreads) {
                const int m = i / klen, k = i - m * klen;
                *reinterpret_cast<uint16_t *>(xs + m * xrowb + 2 * k) = ldg_u16(X + m * ldx + k0 + k);
            }
            __syncthreads();
        }

        // ---- this warp's steps of the chunk, NB - 1 batches in flight
        // (load and compute skip steps past the chunk; batches add in order)
        if constexpr (NB == 3) {
            for (int j0 = 0; part + P * j0 < nsteps; j0 += 3 * kU) {
                load(A0[2], A1[2], k0, nsteps, j0 + 2 * kU);
                compute(A0[0], A1[0], nsteps, j0);
                load(A0[0], A1[0], k0, nsteps, j0 + 3 * kU);
                if (part + P * (j0 + kU) < nsteps) compute(A0[1], A1[1], nsteps, j0 + kU);
                load(A0[1], A1[1], k0, nsteps, j0 + 4 * kU);
                if (part + P * (j0 + 2 * kU) < nsteps) compute(A0[2], A1[2], nsteps, j0 + 2 * kU);
            }
        } else {
            for (int j0 = 0; part + P * j0 < nsteps; j0 += 2 * kU) {
                if (part + P * (j0 + kU) < nsteps) load(A0[1], A1[1], k0, nsteps, j0 + kU);
                compute(A0[0], A1[0], nsteps, j0);
                if (part + P * (j0 + 2 * kU) < nsteps) load(A0[0], A1[0], k0, nsteps, j0 + 2 * kU);
                if (part + P * (j0 + kU) < nsteps) compute(A0[1], A1[1], nsteps, j0 + kU);
            }
        }
    }

    if (late) griddep_launch_dependents();   // every W load of this thread has been issued
    // ---- fragments to shared memory: thread (g, t) holds rows g, g+8 for
    // tokens 2t, 2t+1 of each n8 tile; then the P parts of a tile in order
#pragma unroll
    for (int h = 0; h < NT; ++h)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int tok = 8 * h + 2 * t + (q & 1);
            const int row = g + 8 * (q >> 1);
            red[((tile * P + part) * 16 + row) * MT + tok] = macc[h][q];
        }
    __syncthreads();
    if (S > 1) cluster_wait();             // phase 0: every peer has started
    for (int i = tid; i < RT * 16 * M; i += kDotThreads) {
        const int tl = i / (16 * M), rem = i - tl * 16 * M;
        const int row = rem / M, m = rem - row * M;
        const int n = (blk * RT + tl) * 16 + row;
        if (n < N) {
            float v = red[((tl * P + 0) * 16 + row) * MT + m];
#pragma unroll
            for (int pp = 1; pp < P; ++pp) v += red[((tl * P + pp) * 16 + row) * MT + m];
            if (S == 1) {
                store_y(Y, out_bf16, m * ldy + n, v);
            } else {
                const int c = tl * 16 + row;                     // column within the block
                const uint32_t local = smem_u32(slots + (rank * RT * 16 + c) * MT + m);
                st_shared_cluster_f32(mapa_shared(local, (uint32_t)(c % S)), v);
            }
        }
    }
    if (S > 1) {
        cluster_arrive_release();          // phase 1: the partials are in their owners' slots
        cluster_wait_acquire();
        for (int i = tid; i < RT * 16 * M; i += kDotThreads) {
            const int c = i / M, m = i - c * M;
            const int n = blk * RT * 16 + c;
            if (c % S == rank && n < N) {
                float v = slots[c * MT + m];
                for (int r = 1; r < S; ++r) v += slots[(r * RT * 16 + c) * MT + m];
                store_y(Y, out_bf16, m * ldy + n, v);
            }
        }
    }
}

using MmaKernel = void (*)(const uint16_t *, int64_t, const uint16_t *, int64_t, void *, int64_t,
                           int, int, int, int, int, int *, uint64_t, int, int, int);

// token buckets 8 / 16 / 32 / 64 (M = 17..64: the medium-M regime on large weights)
const MmaKernel kTable[4][3] = {
    {&dotmma_kernel<8, 1>, &dotmma_kernel<8, 2>, &dotmma_kernel<8, 4>},
    {&dotmma_kernel<16, 1>, &dotmma_kernel<16, 2>, &dotmma_kernel<16, 4>},
    {&dotmma_kernel<32, 1>, &dotmma_kernel<32, 2>, &dotmma_kernel<32, 4>},
    {&dotmma_kernel<64, 1>, &dotmma_kernel<64, 2>, &dotmma_kernel<64, 4>}};

int bucket(int M) { return M <= 8 ? 0 : M <= 16 ? 1 : M <= 32 ? 2 : 3; }

int rt_index(int block_n) {
    switch (block_n) { case 16: return 0; case 32: return 1; case 64: return 2; default: return -1; }
}

}  // namespace

bool dotmma_supported(int M, int block_n) { return M >= 1 && M <= kMaxMSplitMma && rt_index(block_n) >= 0; }

int dotmma_tokens(int M) { return 8 << bucket(M); }

int dotmma_smem_bytes(int M, int block_n, int k_chunk, int split_k) {
    const int MT = dotmma_tokens(M);
    return MT * xrow_bytes(k_chunk) + kWarps * 16 * MT * 4 + (split_k > 1 ? split_k * block_n * MT * 4 : 0);
}

cudaError_t dotmma_prepare() {
    for (int a = 0; a < 4; ++a)
        for (int b = 0; b < 3; ++b) {
            cudaError_t e = set_max_dyn_smem(kTable[a][b]);
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

cudaError_t launch_dotmma(const GemmArgs &a, const skinny_plan_t &p, const LaunchCtx &c) {
    const int ri = rt_index(p.block_n);
    const int S = p.split_k;
    if (ri < 0 || a.M < 1 || a.M > kMaxMSplitMma || a.K % 32 != 0 || p.k_chunk % 32 != 0 || p.k_chunk < 32 ||
        !dotmma_split_ok(a.M, a.K, S))
        return cudaErrorInvalidValue;
    const int blocks = (a.N + p.block_n - 1) / p.block_n;
    if ((S == 1 && (p.grid_x != blocks || p.grid_y != 1)) || (S > 1 && (p.grid_x != S || p.grid_y != blocks)) ||
        p.smem_bytes < dotmma_smem_bytes(a.M, p.block_n, p.k_chunk, S))
        return cudaErrorInvalidValue;
    MmaKernel fn = kTable[bucket(a.M)][ri];
    const int x_vec16 = ((reinterpret_cast<uintptr_t>(a.X) & 15) == 0 && (a.ldx & 7) == 0) ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid_x, p.grid_y, 1);
    cfg.blockDim = dim3(kDotThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem_bytes;
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
    return cudaLaunchKernelEx(&cfg, fn, a.X, a.ldx, a.W, a.ldw, a.Y, a.ldy, a.M, a.N, a.K, p.k_chunk, x_vec16,
                              c.status, c.budget_ns, a.out_bf16, S, c.late ? 1 : 0);
}

}  // namespace skinny
