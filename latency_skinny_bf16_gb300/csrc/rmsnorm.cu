// rmsnorm.cu -- the query RMS norm in front of the q_b projection.
//
// Design source: "GLM-5.2 Blackwell decode optimizations", section
// "Implementation breakdown" item 2 and the fused_norm_rope snippet (its
// pid == 2 branch: q_c = _rms_norm(q_c, q_rms_norm_w, eps, Q_DIM), stored to
// q_c_out), whose result is the X of the q_b bf16_skinny_gemm (item 3).
//
// GB300 form.  One CTA of 128 threads per token: the sum of squares in fp32
// (thread j takes the 8-element chunks j, j + 128, ... in ascending k, then a
// warp butterfly and the warps in order: a fixed order, so the result is
// bit-identical run to run, and the same order the fused tcgen05 prologue
// uses), r = 1 / sqrtf(mean + eps) (IEEE square root and division), then
// xn = bf16_rn(x * r * g) written to the
// caller's buffer, which the q_b GEMM launched right behind it reads as X.
// With PDL the kernel lets its dependent launch at once, so the GEMM streams
// its weights while the norm runs and reads xn after griddepcontrol.wait.
#include "common.cuh"
#include "internal.h"

namespace skinny {
namespace {

constexpr int kNormThreads = 128;

__global__ void __launch_bounds__(kNormThreads)
rmsnorm_kernel(const uint16_t *__restrict__ X, int64_t ldx, const uint16_t *__restrict__ G, float eps, int K,
               uint16_t *__restrict__ XN, int64_t ldxn)
{
    __shared__ float part[kNormThreads / 32];
    __shared__ float rstat;
    const int m = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    griddep_launch_dependents();   // the GEMM behind may start streaming its weights now
    griddep_wait();                // X comes from the preceding kernel
    const uint16_t *xm = X + (int64_t)m * ldx;
    const bool vec = (reinterpret_cast<uintptr_t>(xm) & 15) == 0;
    const int chunks = (K + 7) / 8;
    // thread j: the squares of its 8-element chunks c = j, j + 128, ... in
    // ascending k (one fused multiply-add each); the order does not depend on
    // how the chunk is loaded
    float ss = 0.f;
    for (int c = tid; c < chunks; c += kNormThreads) {
        const int k0 = 8 * c;
        if (vec && k0 + 8 <= K) {
            const uint4 q = ldg_v4(xm + k0);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float a = bf16_lo(w[e]), b = bf16_hi(w[e]);
                ss = fmaf(a, a, ss);
                ss = fmaf(b, b, ss);
            }
        } else {
            for (int k = k0; k < min(K, k0 + 8); ++k) {
                const float v = bf16_one(ldg_u16(xm + k));
                ss = fmaf(v, v, ss);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if (lane == 0) part[warp] = ss;
    __syncthreads();
    if (tid == 0) {
        float t = part[0];
        for (int w = 1; w < kNormThreads / 32; ++w) t += part[w];
        rstat = 1.0f / sqrtf(t / (float)K + eps);
    }
    __syncthreads();
    const float r = rstat;
    uint16_t *out = XN + (int64_t)m * ldxn;
    for (int k = tid; k < K; k += kNormThreads)
        out[k] = f32_to_bf16_rn(bf16_one(ldg_u16(xm + k)) * r * bf16_one(ldg_u16(G + k)));
}

}  // namespace

cudaError_t launch_rmsnorm(const uint16_t *X, int64_t ldx, const uint16_t *G, float eps, int M, int K, uint16_t *XN,
                           int64_t ldxn, cudaStream_t stream, bool pdl) {
    if (M < 1 || K < 1) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)M, 1, 1);
    cfg.blockDim = dim3(kNormThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, rmsnorm_kernel, X, ldx, G, eps, K, XN, ldxn);
}

}  // namespace skinny
