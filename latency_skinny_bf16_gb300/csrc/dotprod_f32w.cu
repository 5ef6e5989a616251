// dotprod_f32w.cu -- the dot-product backend for fp32 router weights.
//
// Design source: the dot-product kernel of "[Perf][Feat] Add generic cuteDSL
// LL BF16 router (GEMM)", section "Implementation breakdown" item 1, for the
// router GEMM of models that keep fp32 router weights ("GLM-5.2 Blackwell
// decode optimizations", the linked "FP32 router GEMM shape support and
// tuning" and "Preserve FP32 router weights" changes), and the review note that
// fp32 weights must not be sent to the bf16 kernel.
//
// GB300 form: the bf16 dot-product kernel's layout (a CTA of 128 threads owns
// BN rows of W and the whole K; X[0:M, chunk] staged once in shared memory,
// by bulk async copies when its rows are 16-byte aligned; W streamed straight
// from HBM with non-allocating loads, two batches in flight; fp32 fused
// multiply-add; butterfly + fixed-order cross-warp reduction, so results are
// bit-identical run to run), with W read as fp32 vectors of VW = 4 (128-bit),
// 2 or 1 elements.  W traffic is 4NK bytes.  A bf16 x fp32 product is not
// exact in fp32; each fmaf rounds once, like the bf16 path's sums.
#include "common.cuh"
#include "internal.h"

namespace skinny {
namespace {

constexpr int kWarps = kDotThreads / 32;

template <int VW> struct RawF { float f[VW]; };

template <int VW>
__device__ __forceinline__ RawF<VW> load_wf(const float *p) {
    RawF<VW> r;
    if constexpr (VW == 4) {
        const uint4 v = ldg_stream_v4(p);
        r.f[0] = __uint_as_float(v.x); r.f[1] = __uint_as_float(v.y);
        r.f[2] = __uint_as_float(v.z); r.f[3] = __uint_as_float(v.w);
    } else if constexpr (VW == 2) {
        const uint2 v = ldg_stream_v2(p);
        r.f[0] = __uint_as_float(v.x); r.f[1] = __uint_as_float(v.y);
    } else {
        r.f[0] = __uint_as_float(ldg_stream_u32(p));
    }
    return r;
}

// VW bf16 of X from shared memory (8-byte aligned for VW = 4)
template <int VW>
__device__ __forceinline__ void load_x(const uint16_t *p, float (&f)[VW]) {
    if constexpr (VW == 4) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    } else if constexpr (VW == 2) {
        const uint32_t v = *reinterpret_cast<const uint32_t *>(p);
        f[0] = bf16_lo(v); f[1] = bf16_hi(v);
    } else {
        f[0] = bf16_one(*p);
    }
}

template <int MT, int VW, int BN>
__device__ __forceinline__ void fma_f(float (&acc)[MT][BN], const uint16_t *xs, int kc, int koff,
                                      const RawF<VW> (&w)[BN]) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        float x[VW];
        load_x<VW>(xs + m * kc + koff, x);
#pragma unroll
        for (int e = 0; e < VW; ++e)
#pragma unroll
            for (int r = 0; r < BN; ++r) acc[m][r] = fmaf(x[e], w[r].f[e], acc[m][r]);
    }
}

template <int MT, int VW, int BN>
__global__ void __launch_bounds__(kDotThreads)
dotprod_f32w_kernel(const uint16_t *__restrict__ X, int64_t ldx,
                    const float *__restrict__ W, int64_t ldw,
                    float *__restrict__ Y, int64_t ldy,
                    int N, int K, int kc, int x_vec16, int *status, uint64_t budget_ns)
{
    constexpr int U = (BN >= 4) ? 2 : 8 / BN;      // vectors per row per batch
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem_raw);                          // [MT][kc]
    float *red = reinterpret_cast<float *>(smem_raw + ((MT * kc * 2 + 15) & ~15));   // [kWarps][MT][BN]
    __shared__ __align__(8) uint64_t xbar_storage;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n0 = blockIdx.x * BN;
    const uint32_t xbar = smem_u32(&xbar_storage);
    if (tid == 0) {
        mbar_init(xbar, 1);
        fence_mbarrier_init_cluster();
    }
    __syncthreads();

    const float *wrow[BN];
#pragma unroll
    for (int r = 0; r < BN; ++r) wrow[r] = W + (int64_t)min(n0 + r, N - 1) * ldw;   // rows past N: dropped
    // PDL prologue: this CTA's W rows toward L2 (one prefetch per 128-byte line)
#pragma unroll
    for (int r = 0; r < BN; ++r)
        if (n0 + r < N)
            for (int off = tid * 32; off < K; off += kDotThreads * 32) prefetch_l2(wrow[r] + off);

    float acc[MT][BN];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < BN; ++r) acc[m][r] = 0.f;

    RawF<VW> rawA[U][BN], rawB[U][BN];
    auto load_batch = [&](RawF<VW> (&raw)[U][BN], int k0, int nvec, int v0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + u * kDotThreads;
            if (v < nvec) {
#pragma unroll
                for (int r = 0; r < BN; ++r) raw[u][r] = load_wf<VW>(wrow[r] + k0 + v * VW);
            }
        }
    };
    auto fma_batch = [&](const RawF<VW> (&raw)[U][BN], int nvec, int v0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + u * kDotThreads;
            if (v < nvec) fma_f<MT, VW, BN>(acc, xs, kc, v * VW, raw[u]);
        }
    };
    load_batch(rawA, 0, min(kc, K) / VW, tid);
    griddep_wait();
    griddep_launch_dependents();

    for (int k0 = 0; k0 < K; k0 += kc) {
        const int klen = min(kc, K - k0);
        const int nvec = klen / VW;
        if (k0 > 0) {
            __syncthreads();                     // the previous chunk of X is no longer read
            load_batch(rawA, k0, nvec, tid);
        }
        // ---- X[0:M, k0:k0+klen] into shared memory (bulk copies for the multiple-of-8 part)
        const int kb = x_vec16 ? (klen & ~7) : 0;
        if (x_vec16 && warp == 0) {
            if (lane == 0) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(xbar, (uint32_t)(MT * kb * 2));
            }
            __syncwarp();
            if (kb > 0 && lane < MT)
                bulk_copy_g2s(smem_u32(xs + lane * kc), X + lane * ldx + k0, (uint32_t)(kb * 2), xbar);
        }
        {
            const int rem = klen - kb;
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

        // ---- main part: two batches in flight
        constexpr int kStep = U * kDotThreads;
        if constexpr (MT * BN <= 32) {
            for (int v0 = tid; v0 < nvec; v0 += 2 * kStep) {
                if (v0 + kStep < nvec) load_batch(rawB, k0, nvec, v0 + kStep);
                fma_batch(rawA, nvec, v0);
                if (v0 + 2 * kStep < nvec) load_batch(rawA, k0, nvec, v0 + 2 * kStep);
                if (v0 + kStep < nvec) fma_batch(rawB, nvec, v0 + kStep);
            }
        } else {
            for (int v0 = tid; v0 < nvec; v0 += kStep) {
                if (v0 != tid) load_batch(rawA, k0, nvec, v0);
                fma_batch(rawA, nvec, v0);
            }
        }
        // ---- tail: klen % VW scalars
        const int e0 = nvec * VW;
        if (tid < klen - e0) {
            const int e = e0 + tid;
            RawF<1> t[BN];
#pragma unroll
            for (int r = 0; r < BN; ++r) t[r] = load_wf<1>(wrow[r] + k0 + e);
            fma_f<MT, 1, BN>(acc, xs, kc, e, t);
        }
    }

    // ---- reduction: butterfly in the warp, then the warps in order
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
            Y[m * ldy + n] = s;
        }
    }
}

using F32Kernel = void (*)(const uint16_t *, int64_t, const float *, int64_t, float *, int64_t, int, int, int, int,
                           int *, uint64_t);
template <int MT, int VW, int BN> constexpr F32Kernel kf() { return &dotprod_f32w_kernel<MT, VW, BN>; }

// per M: VW = 4 with BN in {1, 2, 4}; VW in {2, 1} with BN = 1
constexpr int kF32Variants = 5;
template <int MT> struct RowF {
    static constexpr F32Kernel k[kF32Variants] = {kf<MT, 4, 1>(), kf<MT, 4, 2>(), kf<MT, 4, 4>(), kf<MT, 2, 1>(),
                                                  kf<MT, 1, 1>()};
};
const F32Kernel *kTableF[kMaxMSmall] = {
    RowF<1>::k, RowF<2>::k, RowF<3>::k, RowF<4>::k, RowF<5>::k, RowF<6>::k, RowF<7>::k, RowF<8>::k,
    RowF<9>::k, RowF<10>::k, RowF<11>::k, RowF<12>::k, RowF<13>::k, RowF<14>::k, RowF<15>::k, RowF<16>::k};

int f32_variant(int vw, int bn) {
    if (vw == 4) return bn == 1 ? 0 : bn == 2 ? 1 : bn == 4 ? 2 : -1;
    if (bn != 1) return -1;
    return vw == 2 ? 3 : vw == 1 ? 4 : -1;
}

}  // namespace

bool dotprod_f32w_supported(int M, int vec_elems, int block_n) {
    return M >= 1 && M <= kMaxMSmall && f32_variant(vec_elems, block_n) >= 0;
}

int dotprod_f32w_smem_bytes(int M, int block_n, int k_chunk) {
    return ((M * k_chunk * 2 + 15) & ~15) + kWarps * M * block_n * 4;
}

cudaError_t dotprod_f32w_prepare() {
    for (int m = 0; m < kMaxMSmall; ++m)
        for (int v = 0; v < kF32Variants; ++v) {
            cudaError_t e = set_max_dyn_smem(kTableF[m][v]);
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

cudaError_t launch_dotprod_f32w(const uint16_t *X, int64_t ldx, const float *W, int64_t ldw, float *Y, int64_t ldy,
                                int M, int N, int K, const skinny_plan_t &p, const LaunchCtx &c) {
    const int vi = f32_variant(p.vec_elems, p.block_n);
    if (vi < 0 || M < 1 || M > kMaxMSmall || p.k_chunk % 8) return cudaErrorInvalidValue;
    F32Kernel fn = kTableF[M - 1][vi];
    const int x_vec16 = ((reinterpret_cast<uintptr_t>(X) & 15) == 0 && (ldx & 7) == 0) ? 1 : 0;
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
    return cudaLaunchKernelEx(&cfg, fn, X, ldx, W, ldw, Y, ldy, N, K, p.k_chunk, x_vec16, c.status, c.budget_ns);
}

}  // namespace skinny
