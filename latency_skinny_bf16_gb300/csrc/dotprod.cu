// dotprod.cu -- the dot-product backend of the skinny BF16 GEMM.
//
// Design source: "[Perf][Feat] Add generic cuteDSL LL BF16 router (GEMM)",
// section "Implementation breakdown" item 1 (one CTA per expert, unrolled K
// loop of 128-bit loads, warp-shuffle + shared-memory reduction) and the
// _ll_bf16_dotprod.py snippet (K split into a 128-bit main part, a 64-bit tail
// and a scalar remainder; W widened to fp32 and multiply-added per token).
//
// GB300 form.  A CTA of 128 threads owns BN consecutive output columns
// (rows of W) and the whole K.  X[0:M, k-chunk] is staged once per chunk in
// shared memory (the whole K when it fits the budget) and is re-used by the BN
// rows; W is streamed straight from HBM into registers with non-allocating
// read-only loads whose width VW (8/4/2/1 bf16) is the widest that the W base
// pointer and ldw allow for every row, so odd strides never fault and aligned
// ones get 128-bit loads.  Threads stride over K vectors (coalesced: a warp
// reads 32 consecutive vectors of a row), multiply-add in fp32 into
// acc[M][BN] registers, then the partials are reduced by a butterfly shuffle
// in each warp and summed across the 4 warps in shared memory in a fixed
// order, so a plan's result is bit-identical from run to run.
//
// With PDL the CTA warms L2 with its own W rows and puts its first batch of W
// loads in flight (W is a weight, never written by the preceding kernel), then
// waits on griddepcontrol before reading X.  X rows that are 16-byte aligned
// arrive by bulk async copies (the TMA engine, one per row, all in flight at
// once) completing on an mbarrier whose wait is bounded; otherwise threads
// stage X with ordinary L2 loads.
#include "common.cuh"
#include "internal.h"

namespace skinny {
namespace {

constexpr int kWarps = kDotThreads / 32;

// Raw W vector of VW bf16: held as 32-bit words (or one 16-bit value).
template <int VW> struct RawW { uint32_t w[VW / 2]; };
template <> struct RawW<1> { uint16_t h; };

template <int VW>
__device__ __forceinline__ RawW<VW> load_w(const uint16_t *p) {
    RawW<VW> r;
    if constexpr (VW == 8) {
        uint4 v = ldg_stream_v4(p);
        r.w[0] = v.x; r.w[1] = v.y; r.w[2] = v.z; r.w[3] = v.w;
    } else if constexpr (VW == 4) {
        uint2 v = ldg_stream_v2(p);
        r.w[0] = v.x; r.w[1] = v.y;
    } else if constexpr (VW == 2) {
        r.w[0] = ldg_stream_u32(p);
    } else {
        r.h = ldg_stream_u16(p);
    }
    return r;
}

template <int VW>
__device__ __forceinline__ void widen(const RawW<VW> &r, float (&f)[VW]) {
    if constexpr (VW == 1) {
        f[0] = bf16_one(r.h);
    } else {
#pragma unroll
        for (int i = 0; i < VW / 2; ++i) {
            f[2 * i] = bf16_lo(r.w[i]);
            f[2 * i + 1] = bf16_hi(r.w[i]);
        }
    }
}

// X vector of VW bf16 from shared memory (16-byte aligned for VW = 8).
template <int VW>
__device__ __forceinline__ void load_x_smem(const uint16_t *p, float (&f)[VW]) {
    if constexpr (VW == 8) {
        uint4 v = *reinterpret_cast<const uint4 *>(p);
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    } else if constexpr (VW == 4) {
        uint2 v = *reinterpret_cast<const uint2 *>(p);
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    } else if constexpr (VW == 2) {
        uint32_t v = *reinterpret_cast<const uint32_t *>(p);
        f[0] = bf16_lo(v); f[1] = bf16_hi(v);
    } else {
        f[0] = bf16_one(*p);
    }
}

template <int MT, int VW, int BN>
__device__ __forceinline__ void fma_vec(float (&acc)[MT][BN], const uint16_t *xs, int kc, int koff,
                                        const RawW<VW> (&raw)[BN]) {
    float w[BN][VW];
#pragma unroll
    for (int r = 0; r < BN; ++r) widen<VW>(raw[r], w[r]);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        float x[VW];
        load_x_smem<VW>(xs + m * kc + koff, x);
#pragma unroll
        for (int e = 0; e < VW; ++e)
#pragma unroll
            for (int r = 0; r < BN; ++r) acc[m][r] = fmaf(x[e], w[r][e], acc[m][r]);
    }
}

template <int MT, int VW, int BN>
__global__ void __launch_bounds__(kDotThreads)
dotprod_kernel(const uint16_t *__restrict__ X, int64_t ldx,
               const uint16_t *__restrict__ W, int64_t ldw,
               void *__restrict__ Y, int64_t ldy,
               int N, int K, int kc, int x_vec16, int *status, uint64_t budget_ns, int out_bf16, int late)
{
    // Loads in flight per thread per step: U vectors of each of the BN rows.
    constexpr int U = (BN >= 8) ? 1 : 8 / BN;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem_raw);                       // [MT][kc]
    float *red = reinterpret_cast<float *>(smem_raw + ((MT * kc * 2 + 15) & ~15));  // [kWarps][MT][BN]

    __shared__ __align__(8) uint64_t xbar_storage;   // X chunk copies complete here
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n0 = blockIdx.x * BN;
    const uint32_t xbar = smem_u32(&xbar_storage);
    if (tid == 0) {
        mbar_init(xbar, 1);
        fence_mbarrier_init_cluster();
    }
    __syncthreads();

    const uint16_t *wrow[BN];
#pragma unroll
    for (int r = 0; r < BN; ++r) {
        const int n = min(n0 + r, N - 1);   // rows past N re-read row N-1; their sums are dropped
        wrow[r] = W + (int64_t)n * ldw;
    }

    // PDL prologue: pull this CTA's W rows toward L2 while the preceding
    // kernel drains (one prefetch per 128-byte line), and put the first batch
    // of W vectors in flight before X is needed.  W is a weight, never
    // written by the preceding kernel; X is read only after griddepcontrol.wait.
#pragma unroll
    for (int r = 0; r < BN; ++r)
        if (n0 + r < N)
            for (int off = tid * 64; off < K; off += kDotThreads * 64) prefetch_l2(wrow[r] + off);

    float acc[MT][BN];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < BN; ++r) acc[m][r] = 0.f;

    // Batch b of a chunk: vectors v = tid + (b*U + u) * T, u < U, predicated.
    // Two register buffers: batch b+1 is in flight while batch b is consumed.
    RawW<VW> rawA[U][BN], rawB[U][BN];
    auto load_batch = [&](RawW<VW> (&raw)[U][BN], int k0, int nvec, int v0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + u * kDotThreads;
            if (v < nvec) {
#pragma unroll
                for (int r = 0; r < BN; ++r) raw[u][r] = load_w<VW>(wrow[r] + k0 + v * VW);
            }
        }
    };
    auto fma_batch = [&](const RawW<VW> (&raw)[U][BN], int nvec, int v0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + u * kDotThreads;
            if (v < nvec) fma_vec<MT, VW, BN>(acc, xs, kc, v * VW, raw[u]);
        }
    };
    {
        const int klen0 = min(kc, K);
        load_batch(rawA, 0, klen0 / VW, tid);
    }
    griddep_wait();
    if (!late) griddep_launch_dependents();

    for (int k0 = 0; k0 < K; k0 += kc) {
        const int klen = min(kc, K - k0);
        const int nvec = klen / VW;
        if (k0 > 0) {
            __syncthreads();            // every thread is done with the previous chunk of X
            load_batch(rawA, k0, nvec, tid);  // first W batch of this chunk, before staging X
        }
        // ---- stage X[0:M, k0:k0+klen] in shared memory: when X rows are
        // 16-byte aligned, one bulk async copy per row (the TMA engine) for
        // the whole multiple-of-8 part, the last klen % 8 elements by hand
        const int kb = x_vec16 ? (klen & ~7) : 0;
        if (x_vec16 && warp == 0) {
            if (lane == 0) {
                fence_proxy_async_smem();   // the previous chunk was read by ordinary loads
                mbar_arrive_expect_tx(xbar, (uint32_t)(MT * kb * 2));
            }
            __syncwarp();
            if (kb > 0 && lane < MT)
                bulk_copy_g2s(smem_u32(xs + lane * kc), X + lane * ldx + k0, (uint32_t)(kb * 2), xbar);
        }
        {
            const int rem = klen - kb;
#pragma unroll 4
            for (int i = tid; i < MT * rem; i += kDotThreads) {
                const int m = i / rem, k = kb + (i - m * rem);
                xs[m * kc + k] = ldg_u16(X + m * ldx + k0 + k);
            }
        }
        __syncthreads();
        if (x_vec16) {
            const uint32_t par = (uint32_t)((k0 / kc) & 1);
            if (!mbar_wait_bounded(xbar, par, budget_ns)) {
                if (lane == 0) report_status(status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitX);
                if (!mbar_wait_bounded(xbar, par, 200ull * 1000 * 1000) && lane == 0)
                    report_status(status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitDrain);
            }
        }

        // ---- main part: VW-wide vectors, U per row per batch, two batches in flight
        constexpr int kStep = U * kDotThreads;
        if constexpr (MT * BN <= 32) {
            for (int v0 = tid; v0 < nvec; v0 += 2 * kStep) {
                if (v0 + kStep < nvec) load_batch(rawB, k0, nvec, v0 + kStep);
                fma_batch(rawA, nvec, v0);
                if (v0 + 2 * kStep < nvec) load_batch(rawA, k0, nvec, v0 + 2 * kStep);
                if (v0 + kStep < nvec) fma_batch(rawB, nvec, v0 + kStep);
            }
        } else {
            // many accumulators: one register buffer (no spills)
            for (int v0 = tid; v0 < nvec; v0 += kStep) {
                if (v0 != tid) load_batch(rawA, k0, nvec, v0);
                fma_batch(rawA, nvec, v0);
            }
        }

        // ---- tail: klen % VW elements (only the last chunk has one).  With
        // 128-bit main loads a 64-bit step takes 4 of them, then scalars.
        const int e0 = nvec * VW;
        const int tail = klen - e0;
        if (tail > 0) {
            if (VW == 8 && tail >= 4) {
                if (tid == 0) {
                    RawW<4> t4[BN];
#pragma unroll
                    for (int r = 0; r < BN; ++r) t4[r] = load_w<4>(wrow[r] + k0 + e0);
                    fma_vec<MT, 4, BN>(acc, xs, kc, e0, t4);
                } else if (tid <= tail - 4) {
                    const int e = e0 + 4 + (tid - 1);
                    RawW<1> t1[BN];
#pragma unroll
                    for (int r = 0; r < BN; ++r) t1[r] = load_w<1>(wrow[r] + k0 + e);
                    fma_vec<MT, 1, BN>(acc, xs, kc, e, t1);
                }
            } else if (tid < tail) {
                const int e = e0 + tid;
                RawW<1> t1[BN];
#pragma unroll
                for (int r = 0; r < BN; ++r) t1[r] = load_w<1>(wrow[r] + k0 + e);
                fma_vec<MT, 1, BN>(acc, xs, kc, e, t1);
            }
        }
    }

    if (late) griddep_launch_dependents();   // every W load of this thread has been issued
    // ---- reduction: butterfly in the warp, then the 4 warps in order 0..3
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < BN; ++r) {
            float s = acc[m][r];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
            acc[m][r] = s;
        }
    if (lane == 0) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int r = 0; r < BN; ++r) red[(warp * MT + m) * BN + r] = acc[m][r];
    }
    __syncthreads();
    for (int i = tid; i < MT * BN; i += kDotThreads) {
        const int m = i / BN, r = i - m * BN;
        const int n = n0 + r;
        if (n < N) {
            float s = red[m * BN + r];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) s += red[(w * MT + m) * BN + r];
            store_y(Y, out_bf16, m * ldy + n, s);
        }
    }
}

// ------------------------------------------------------------------ instantiation table
using DotKernel = void (*)(const uint16_t *, int64_t, const uint16_t *, int64_t, void *, int64_t,
                           int, int, int, int, int *, uint64_t, int, int);

template <int MT, int VW, int BN> constexpr DotKernel kfn() { return &dotprod_kernel<MT, VW, BN>; }

// Per M: VW=8 with BN in {1,2,4,8}; VW in {4,2,1} with BN = 1.
constexpr int kDotVariants = 7;
template <int MT> struct Row {
    static constexpr DotKernel k[kDotVariants] = {
        kfn<MT, 8, 1>(), kfn<MT, 8, 2>(), kfn<MT, 8, 4>(), kfn<MT, 8, 8>(),
        kfn<MT, 4, 1>(), kfn<MT, 2, 1>(), kfn<MT, 1, 1>()};
};

const DotKernel *kTable[kMaxMSmall] = {
    Row<1>::k, Row<2>::k, Row<3>::k, Row<4>::k, Row<5>::k, Row<6>::k, Row<7>::k, Row<8>::k,
    Row<9>::k, Row<10>::k, Row<11>::k, Row<12>::k, Row<13>::k, Row<14>::k, Row<15>::k, Row<16>::k};

int variant_index(int vec_elems, int block_n) {
    if (vec_elems == 8) {
        switch (block_n) { case 1: return 0; case 2: return 1; case 4: return 2; case 8: return 3; default: return -1; }
    }
    if (block_n != 1) return -1;
    switch (vec_elems) { case 4: return 4; case 2: return 5; case 1: return 6; default: return -1; }
}

}  // namespace

bool dotprod_supported(int M, int vec_elems, int block_n) {
    return M >= 1 && M <= kMaxMSmall && variant_index(vec_elems, block_n) >= 0;
}

int dotprod_smem_bytes(int M, int block_n, int k_chunk) {
    return ((M * k_chunk * 2 + 15) & ~15) + kWarps * M * block_n * 4;
}

cudaError_t dotprod_prepare() {
    for (int m = 0; m < kMaxMSmall; ++m)
        for (int v = 0; v < kDotVariants; ++v) {
            cudaError_t e = set_max_dyn_smem(kTable[m][v]);
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

cudaError_t launch_dotprod(const GemmArgs &a, const skinny_plan_t &p, const LaunchCtx &c) {
    const int vi = variant_index(p.vec_elems, p.block_n);
    if (vi < 0 || a.M < 1 || a.M > kMaxMSmall) return cudaErrorInvalidValue;
    DotKernel fn = kTable[a.M - 1][vi];
    const int x_vec16 = ((reinterpret_cast<uintptr_t>(a.X) & 15) == 0 && (a.ldx & 7) == 0) ? 1 : 0;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid_x, 1, 1);
    cfg.blockDim = dim3(kDotThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = c.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, a.X, a.ldx, a.W, a.ldw, a.Y, a.ldy, a.N, a.K, p.k_chunk, x_vec16, c.status,
                              c.budget_ns, a.out_bf16, c.late ? 1 : 0);
}

}  // namespace skinny
