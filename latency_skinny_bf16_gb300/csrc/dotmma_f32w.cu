// dotmma_f32w.cu -- the tensor-core dot-product for fp32 router weights.
//
// Design source: the dot-product kernel of "[Perf][Feat] Add generic cuteDSL
// LL BF16 router (GEMM)", section "Implementation breakdown" item 1 (a CTA
// owns a block of output columns, W streamed with 128-bit loads, partials
// reduced in a fixed order) with item 2's split of K over the CTAs of a
// thread-block cluster and a DSMEM reduction, for the fp32 router weights of
// "GLM-5.2 Blackwell decode optimizations" (the linked "FP32 router GEMM shape
// support and tuning" and "Preserve FP32 router weights" changes).
//
// GB300 form.  The layout is the bf16 tensor-core dot-product's, with NW = 4
// or 8 warps: a CTA owns RT tiles of 16 W rows; warp w takes tile w % RT and
// every P-th 32-element K step (P = NW / RT); with a cluster of S CTAs each CTA takes one
// K slice and sends its partials to the owner CTA of each column through
// st.shared::cluster, and the owner adds the S slots in rank order.  For one
// step, lane (g = lane/4, t = lane%4) loads W[row g][8t .. 8t+7] and
// W[row g+8][8t .. 8t+7] as fp32 (four 128-bit non-allocating loads).
//
// Each weight w is carried as two tf32 terms: hi = w with its 13 low mantissa
// bits cleared, lo = (w - hi) cleared the same way (w - hi is exact in fp32).
// Clearing loses less than 2^-10 of its argument, so |w - hi - lo| is below
// 2^-20 |w|; a bf16 X value is exact in tf32 and a tf32 x tf32 product is
// exact in fp32, so x * w is carried to within 2^-20 of |x * w| (the bar is
// 1e-5 of sum |x * w|).  mma.sync m16n8k8 (tf32 -> fp32) takes the terms: per
// 32-element step 4 MMAs of 8 k for lo, then 4 for hi (the small terms
// first).  MMA j takes physical k = 8t + 2j on the k slot t and 8t + 2j + 1 on
// the slot t + 4, on A (W) and on B (X) alike, so every MMA sums matching
// products.  The split is two masks and a subtraction per weight, no
// conversion instruction: the three-term bf16 split first built here spent
// about 480 dependent instructions per step and ran latency-bound.  Batches of
// 2 steps are double-buffered in registers; each batch's 16 MMAs per token
// tile accumulate in one register sum, then are added into the fp32
// accumulator with a rounded add.  A weight that is not finite is carried
// whole by hi (lo = 0, a NaN as the quiet NaN), so it propagates as in IEEE
// arithmetic; clearing bits never rounds a finite weight up to infinity.
//
// The rank's whole K slice of X (M rows) is resident in shared memory (row
// stride 64 mod 128 bytes, conflict-free 128-bit reads), staged by bulk
// copies when X rows are 16-byte aligned (bounded mbarrier wait), else by
// ordinary loads.  With PDL the first batch of W loads is issued before
// griddepcontrol.wait.  Needs fp32 W rows 16-byte aligned and K % 32 == 0.
#include "common.cuh"
#include "dotmma_f32w.h"

namespace skinny {
namespace {

// Warps per CTA, by token bucket: 8 at 8 tokens (116 registers, two CTAs an
// SM: with K over a cluster of 8 CTAs a router CTA holds 16 rows x 896 fp32,
// and 8 warps x 2 batches of 2 steps put all 57 KB in flight at once), 4 at 16
// tokens (138 registers: 8 warps would leave one CTA an SM, and 16 clusters of
// 8 CTAs would then not all be resident at once).
__host__ __device__ constexpr int f32w_warps(int MT) { return MT == 8 ? 8 : 4; }
constexpr int kUF = 2;   // 32-element K steps per warp per batch

__host__ __device__ inline int xrow_bytes_f(int ks) { return ((ks * 2 + 127) & ~127) + 64; }

__device__ __forceinline__ uint4 lds128_f(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }

// w as hi + lo, both exact tf32 values (fp32 bit patterns)
__device__ __forceinline__ void split_tf32(uint32_t wb, uint32_t &h, uint32_t &l) {
    const uint32_t hb = wb & 0xFFFFE000u;
    const uint32_t lb = __float_as_uint(__uint_as_float(wb) - __uint_as_float(hb)) & 0xFFFFE000u;
    const bool special = (wb & 0x7F800000u) == 0x7F800000u;        // inf or NaN
    h = special ? ((wb & 0x007FFFFFu) ? 0x7FC00000u : wb) : hb;
    l = special ? 0u : lb;
}

// D += A (16 x 8, tf32, row) * B (8 x 8, tf32, col), fp32 accumulate
__device__ __forceinline__ void mma_tf32_1688(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

}  // namespace

// K elements per cluster rank: ceil(K / S) rounded up to a whole 32-element step.
__host__ __device__ int dotmma_f32w_k_slice(int K, int S) { return ((K + S - 1) / S + 31) / 32 * 32; }

bool dotmma_f32w_split_ok(int K, int S) {
    if (S == 1) return true;
    if (S < 1 || S > kSplitMaxCluster) return false;
    return (int64_t)(S - 1) * dotmma_f32w_k_slice(K, S) < K;
}

namespace {

template <int MT, int RT, int NW>
__global__ void __launch_bounds__(NW * 32)
dotmma_f32w_kernel(const uint16_t *__restrict__ X, int64_t ldx,
                   const float *__restrict__ W, int64_t ldw,
                   float *__restrict__ Y, int64_t ldy,
                   int M, int N, int K, int x_vec16, int *status, uint64_t budget_ns, int S, int late)
{
    constexpr int P = NW / RT;        // K parts per row tile
    constexpr int kThreads = NW * 32;
    constexpr int NT = MT / 8;        // n8 token tiles
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t xbar_storage;

    // S > 1: grid S x blocks, this CTA takes K slice `rank` of column block `blk`
    const int rank = (S > 1) ? (int)blockIdx.x : 0;
    const int blk = (S > 1) ? (int)blockIdx.y : (int)blockIdx.x;
    const int KS = (S > 1) ? dotmma_f32w_k_slice(K, S) : K;
    const int kbeg = rank * KS, kend = min(K, kbeg + KS);
    const int klen = max(0, kend - kbeg);
    const int nsteps = klen / 32;
    const int xrowb = xrow_bytes_f(KS);
    uint8_t *xs = smem;                                              // [MT][xrowb]
    float *red = reinterpret_cast<float *>(smem + MT * xrowb);       // [RT][P][16][MT]
    float *slots = red + NW * 16 * MT;                               // S > 1: [S][RT * 16][MT]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tile = warp % RT, part = warp / RT;
    const int g = lane >> 2, t = lane & 3;
    const int n0 = (blk * RT + tile) * 16;
    // rows past N re-read row N-1; their sums are dropped
    const float *w0 = W + (int64_t)min(n0 + g, N - 1) * ldw + kbeg + 8 * t;
    const float *w1 = W + (int64_t)min(n0 + g + 8, N - 1) * ldw + kbeg + 8 * t;
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

    // a batch of kUF steps, steps s = part + P * (j0 + u); per step and lane
    // 8 fp32 of row g (two 128-bit loads) and 8 of row g + 8
    uint4 A0[2][kUF][2], A1[2][kUF][2];
    auto load = [&](uint4 (&a0)[kUF][2], uint4 (&a1)[kUF][2], int j0) {
#pragma unroll
        for (int u = 0; u < kUF; ++u) {
            const int s = part + P * (j0 + u);
            if (s < nsteps) {
                a0[u][0] = ldg_stream_v4(w0 + s * 32);
                a0[u][1] = ldg_stream_v4(w0 + s * 32 + 4);
                a1[u][0] = ldg_stream_v4(w1 + s * 32);
                a1[u][1] = ldg_stream_v4(w1 + s * 32 + 4);
            }
        }
    };
    auto compute = [&](const uint4 (&a0)[kUF][2], const uint4 (&a1)[kUF][2], int j0) {
        float d[NT][4];
#pragma unroll
        for (int h = 0; h < NT; ++h)
#pragma unroll
            for (int q = 0; q < 4; ++q) d[h][q] = 0.f;
#pragma unroll
        for (int u = 0; u < kUF; ++u) {
            const int s = part + P * (j0 + u);
            if (s < nsteps) {
                const uint8_t *xp = xs + g * xrowb + (s * 32 + 8 * t) * 2;
                uint4 xv[NT];
#pragma unroll
                for (int h = 0; h < NT; ++h) xv[h] = lds128_f(xp + h * 8 * xrowb);
                // the 8 weights of row g (r = 0) and of row g + 8 (r = 1), k = 8t + e
                const uint32_t wv[2][8] = {
                    {a0[u][0].x, a0[u][0].y, a0[u][0].z, a0[u][0].w, a0[u][1].x, a0[u][1].y, a0[u][1].z, a0[u][1].w},
                    {a1[u][0].x, a1[u][0].y, a1[u][0].z, a1[u][0].w, a1[u][1].x, a1[u][1].y, a1[u][1].z, a1[u][1].w}};
                uint32_t tm[2][2][8];   // [lo, hi][row][e]
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int e = 0; e < 8; ++e) split_tf32(wv[r][e], tm[1][r][e], tm[0][r][e]);
#pragma unroll
                for (int pt = 0; pt < 2; ++pt)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t fa[4] = {tm[pt][0][2 * j], tm[pt][1][2 * j], tm[pt][0][2 * j + 1],
                                                tm[pt][1][2 * j + 1]};
#pragma unroll
                        for (int h = 0; h < NT; ++h) {
                            const uint32_t xw = j == 0 ? xv[h].x : j == 1 ? xv[h].y : j == 2 ? xv[h].z : xv[h].w;
                            mma_tf32_1688(d[h], fa, xw << 16, xw & 0xFFFF0000u);
                        }
                    }
            }
        }
#pragma unroll
        for (int h = 0; h < NT; ++h)
#pragma unroll
            for (int q = 0; q < 4; ++q) macc[h][q] += d[h][q];
    };

    load(A0[0], A1[0], 0);   // W is a weight: in flight before the PDL wait
    griddep_wait();
    if (!late) griddep_launch_dependents();

    // ---- X[0:M, kbeg:kend] in shared memory (klen is a multiple of 32)
    if (x_vec16) {
        if (warp == 0) {
            if (lane == 0) mbar_arrive_expect_tx(xbar, (uint32_t)(M * klen * 2));
            __syncwarp();
            if (klen > 0)
                for (int r = lane; r < M; r += 32)
                    bulk_copy_g2s(smem_u32(xs + r * xrowb), X + r * ldx + kbeg, (uint32_t)(klen * 2), xbar);
        }
        if (!mbar_wait_bounded(xbar, 0, budget_ns)) {
            if (lane == 0) report_status(status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitX);
            if (!mbar_wait_bounded(xbar, 0, 200ull * 1000 * 1000) && lane == 0)
                report_status(status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitDrain);
        }
    } else {
#pragma unroll 4
        for (int i = tid; i < M * klen; i += kThreads) {
            const int m = i / klen, k = i - m * klen;
            *reinterpret_cast<uint16_t *>(xs + m * xrowb + 2 * k) = ldg_u16(X + m * ldx + kbeg + k);
        }
        __syncthreads();
    }

    // ---- this warp's steps, one batch in flight while the other is consumed
    for (int j0 = 0; part + P * j0 < nsteps; j0 += 2 * kUF) {
        if (part + P * (j0 + kUF) < nsteps) load(A0[1], A1[1], j0 + kUF);
        compute(A0[0], A1[0], j0);
        if (part + P * (j0 + 2 * kUF) < nsteps) load(A0[0], A1[0], j0 + 2 * kUF);
        if (part + P * (j0 + kUF) < nsteps) compute(A0[1], A1[1], j0 + kUF);
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
    for (int i = tid; i < RT * 16 * M; i += kThreads) {
        const int tl = i / (16 * M), rem = i - tl * 16 * M;
        const int row = rem / M, m = rem - row * M;
        const int n = (blk * RT + tl) * 16 + row;
        if (n < N) {
            float v = red[((tl * P + 0) * 16 + row) * MT + m];
#pragma unroll
            for (int pp = 1; pp < P; ++pp) v += red[((tl * P + pp) * 16 + row) * MT + m];
            if (S == 1) {
                Y[m * ldy + n] = v;
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
        for (int i = tid; i < RT * 16 * M; i += kThreads) {
            const int c = i / M, m = i - c * M;
            const int n = blk * RT * 16 + c;
            if (c % S == rank && n < N) {
                float v = slots[c * MT + m];
                for (int r = 1; r < S; ++r) v += slots[(r * RT * 16 + c) * MT + m];
                Y[m * ldy + n] = v;
            }
        }
    }
}

using F32MmaKernel = void (*)(const uint16_t *, int64_t, const float *, int64_t, float *, int64_t, int, int, int, int,
                              int *, uint64_t, int, int);

// token buckets 8 / 16; block_n 16 / 32
const F32MmaKernel kTableFM[2][2] = {
    {&dotmma_f32w_kernel<8, 1, f32w_warps(8)>, &dotmma_f32w_kernel<8, 2, f32w_warps(8)>},
    {&dotmma_f32w_kernel<16, 1, f32w_warps(16)>, &dotmma_f32w_kernel<16, 2, f32w_warps(16)>}};

int rt_index_f(int block_n) { return block_n == 16 ? 0 : block_n == 32 ? 1 : -1; }

}  // namespace


bool dotmma_f32w_supported(int M, int block_n) { return M >= 1 && M <= kMaxMSmall && rt_index_f(block_n) >= 0; }

int dotmma_f32w_threads(int M) { return 32 * f32w_warps(M <= 8 ? 8 : 16); }

int dotmma_f32w_smem_bytes(int M, int block_n, int K, int split_k) {
    const int MT = M <= 8 ? 8 : 16;
    const int ks = split_k > 1 ? dotmma_f32w_k_slice(K, split_k) : K;
    return MT * xrow_bytes_f(ks) + f32w_warps(MT) * 16 * MT * 4 + (split_k > 1 ? split_k * block_n * MT * 4 : 0);
}

cudaError_t dotmma_f32w_prepare() {
    for (int a = 0; a < 2; ++a)
        for (int b = 0; b < 2; ++b) {
            cudaError_t e = set_max_dyn_smem(kTableFM[a][b]);
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

cudaError_t launch_dotmma_f32w(const uint16_t *X, int64_t ldx, const float *W, int64_t ldw, float *Y, int64_t ldy,
                               int M, int N, int K, const skinny_plan_t &p, const LaunchCtx &c) {
    const int ri = rt_index_f(p.block_n);
    const int S = p.split_k;
    if (ri < 0 || M < 1 || M > kMaxMSmall || K < 32 || K % 32 != 0 || !dotmma_f32w_split_ok(K, S) ||
        (reinterpret_cast<uintptr_t>(W) & 15) || (ldw & 3))
        return cudaErrorInvalidValue;
    const int blocks = (N + p.block_n - 1) / p.block_n;
    if (p.threads != dotmma_f32w_threads(M)) return cudaErrorInvalidValue;
    if ((S == 1 && (p.grid_x != blocks || p.grid_y != 1)) || (S > 1 && (p.grid_x != S || p.grid_y != blocks)) ||
        p.smem_bytes < dotmma_f32w_smem_bytes(M, p.block_n, K, S) || p.smem_bytes > kMaxDynSmem)
        return cudaErrorInvalidValue;
    F32MmaKernel fn = kTableFM[M <= 8 ? 0 : 1][ri];
    const int x_vec16 = ((reinterpret_cast<uintptr_t>(X) & 15) == 0 && (ldx & 7) == 0) ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid_x, p.grid_y, 1);
    cfg.blockDim = dim3(p.threads, 1, 1);
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
    return cudaLaunchKernelEx(&cfg, fn, X, ldx, W, ldw, Y, ldy, M, N, K, x_vec16, c.status, c.budget_ns, S,
                              c.late ? 1 : 0);
}

}  // namespace skinny
