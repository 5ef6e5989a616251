// topk.cu -- the router epilogue: softmax over each token's expert logits and
// its top-k experts.
//
// Design source: "[Perf][Feat] Add generic cuteDSL LL BF16 router (GEMM)",
// section "Implementation breakdown" item 4 (the MoE gate's forward consumes
// the router logits).  The pages print no epilogue, so this is the plainest
// one: p = softmax(logits of the token), the k largest logits (equal logits:
// lower index first), weights p of those, optionally renormalised to sum to 1.
//
// GB300 form.  A separate small kernel, launched right after the router GEMM
// on the same stream (with PDL it starts while the GEMM drains and waits for
// it in griddepcontrol.wait): the k largest entries of a token need all N of
// its logits, which the GEMM spreads over many CTAs and clusters.  One CTA of
// 128 threads per token keeps the row in shared memory; the max and the sum
// of exponentials are reduced in a fixed order (per thread ascending, warp
// butterfly, warps in order), and each of the k selections is a block-wide
// argmax over the entries not yet taken, so results are bit-identical from
// run to run.  Rows of at most 1024 logits (the router's 256 / 384 experts)
// take a warp per token instead, the row in registers and no barrier at all.
// expf is CUDA's own.
#include "common.cuh"
#include "internal.h"

namespace skinny {
namespace {

constexpr int kTopkThreads = 128;
constexpr int kTopkWarps = kTopkThreads / 32;

// (v, n) is a better pick than (bv, bn): the larger logit; a NaN ranks below
// every other value (-inf included); equal logits, or two NaNs, the lower
// index.  n < 0 marks "none yet".  Every row thus has a total order, so the k
// ids are distinct valid indices whatever the logits hold.
__device__ __forceinline__ bool better(float v, int n, float bv, int bn) {
    const bool vnan = v != v, bnan = bv != bv;
    const bool gt = !vnan & (bnan | (v > bv));                  // a better value class or value
    const bool eq = (vnan & bnan) | (!vnan & !bnan & (v == bv));
    return (n >= 0) & ((bn < 0) | gt | (eq & (n < bn)));
}

// The same order as one 64-bit key (larger = better): the logit mapped to an
// unsigned integer that grows with it (-0 as +0, every NaN to 0, below -inf),
// then the complement of the index, so equal logits favour the lower index.
// 0 itself is "none": every real candidate's key has its index bits set.
__device__ __forceinline__ uint64_t rank_key(float v, int n) {
    uint32_t b = (v == 0.f) ? 0u : __float_as_uint(v);
    uint32_t o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    if (v != v) o = 0u;
    return ((uint64_t)o << 32) | (uint32_t)~(uint32_t)n;
}
// The logit of a key (a NaN for the NaN class; -0 comes back as +0).
__device__ __forceinline__ float key_value(uint64_t key) {
    const uint32_t o = (uint32_t)(key >> 32);
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

__global__ void __launch_bounds__(kTopkThreads)
router_topk_kernel(const float *__restrict__ L, int64_t ldl, int N, int k, int renormalize,
                   float *__restrict__ weights, int64_t ldwt, int32_t *__restrict__ ids, int64_t ldid)
{
    extern __shared__ __align__(16) uint8_t smem[];
    float *row = reinterpret_cast<float *>(smem);                       // [N]
    uint8_t *taken = smem + (size_t)N * 4;                              // [N]
    __shared__ float wv[kTopkWarps];
    __shared__ int wn[kTopkWarps];
    __shared__ float chosen[kTopkMaxK];
    __shared__ float stat[2];   // max, sum of exponentials
    const int m = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    griddep_wait();   // the logits come from the preceding kernel (the router GEMM)
    const float *src = L + (int64_t)m * ldl;
    float lmax = -INFINITY;
    for (int n = tid; n < N; n += kTopkThreads) {
        const float v = src[n];
        row[n] = v;
        taken[n] = 0;
        lmax = fmaxf(lmax, v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, o));
    if (lane == 0) wv[warp] = lmax;
    __syncthreads();
    if (tid == 0) {
        float v = wv[0];
        for (int w = 1; w < kTopkWarps; ++w) v = fmaxf(v, wv[w]);
        stat[0] = v;
    }
    __syncthreads();
    lmax = stat[0];
    float s = 0.f;
    for (int n = tid; n < N; n += kTopkThreads) s += expf(row[n] - lmax);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    if (lane == 0) wv[warp] = s;
    __syncthreads();
    if (tid == 0) {
        float v = wv[0];
        for (int w = 1; w < kTopkWarps; ++w) v += wv[w];
        stat[1] = v;
    }
    __syncthreads();
    const float denom = stat[1];

    for (int i = 0; i < k; ++i) {
        float bv = -INFINITY;
        int bn = -1;
        for (int n = tid; n < N; n += kTopkThreads)
            if (!taken[n] && better(row[n], n, bv, bn)) { bv = row[n]; bn = n; }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
            const int on = __shfl_xor_sync(0xFFFFFFFFu, bn, o);
            if (better(ov, on, bv, bn)) { bv = ov; bn = on; }
        }
        if (lane == 0) { wv[warp] = bv; wn[warp] = bn; }
        __syncthreads();
        if (tid == 0) {
            float v = wv[0];
            int n = wn[0];
            for (int w = 1; w < kTopkWarps; ++w)
                if (better(wv[w], wn[w], v, n)) { v = wv[w]; n = wn[w]; }
            taken[n] = 1;
            ids[(int64_t)m * ldid + i] = n;
            chosen[i] = expf(row[n] - lmax) / denom;
        }
        __syncthreads();
    }
    if (tid == 0 && renormalize) {
        float t = 0.f;
        for (int i = 0; i < k; ++i) t += chosen[i];
        stat[1] = t;
    }
    __syncthreads();
    griddep_launch_dependents();
    for (int i = tid; i < k; i += kTopkThreads)
        weights[(int64_t)m * ldwt + i] = renormalize ? chosen[i] / stat[1] : chosen[i];
}

// One warp per token for N <= 32 * VPL (VPL <= 32): lane l holds the logits
// n = l + 32 j in registers; the max and the sum of exponentials are warp
// butterflies over per-lane sums in ascending j, and each selection is a warp
// maximum of rank keys over the entries not yet taken: no barrier and no
// shared memory.  Four tokens per CTA.
template <int VPL>
__global__ void __launch_bounds__(kTopkThreads)
router_topk_warp_kernel(const float *__restrict__ L, int64_t ldl, int M, int N, int k, int renormalize,
                        float *__restrict__ weights, int64_t ldwt, int32_t *__restrict__ ids, int64_t ldid)
{
    const int lane = threadIdx.x & 31;
    const int m = blockIdx.x * kTopkWarps + (threadIdx.x >> 5);
    griddep_wait();   // the logits come from the preceding kernel (the router GEMM)
    if (m >= M) return;
    const float *src = L + (int64_t)m * ldl;
    float v[VPL];
    float lmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
        const int n = lane + 32 * j;
        v[j] = (n < N) ? src[n] : -INFINITY;
        if (n < N) lmax = fmaxf(lmax, v[j]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, o));
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < VPL; ++j)
        if (lane + 32 * j < N) s += expf(v[j] - lmax);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    // each selection: the largest key not yet taken, per lane over its VPL
    // keys, then across the warp (64-bit butterfly); the owner lane marks it
    uint64_t key[VPL];
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
        const int n = lane + 32 * j;
        key[j] = (n < N) ? rank_key(v[j], n) : 0ull;
    }
    // lane l keeps choice l (lo) and choice 32 + l (hi); every lane sums the
    // chosen probabilities in selection order
    float p_lo = 0.f, p_hi = 0.f, total = 0.f;
    int id_lo = -1, id_hi = -1;
    for (int i = 0; i < k; ++i) {
        // the lane's largest key: a pairwise tree (depth log2 VPL, not VPL)
        uint64_t t[VPL];
#pragma unroll
        for (int j = 0; j < VPL; ++j) t[j] = key[j];
#pragma unroll
        for (int lvl = 1; lvl < VPL; lvl *= 2)
#pragma unroll
            for (int j = 0; j + lvl < VPL; j += 2 * lvl) t[j] = t[j + lvl] > t[j] ? t[j + lvl] : t[j];
        uint64_t best = t[0];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t other = __shfl_xor_sync(0xFFFFFFFFu, best, o);
            best = other > best ? other : best;
        }
        const int wn = (int)~(uint32_t)best;
        // keys are unique (the index is part of each): clear the winner's
#pragma unroll
        for (int j = 0; j < VPL; ++j) key[j] = (key[j] == best) ? 0ull : key[j];
        const float p = expf(key_value(best) - lmax) / s;
        total += p;
        if (lane == (i & 31)) {
            if (i < 32) { p_lo = p; id_lo = wn; } else { p_hi = p; id_hi = wn; }
        }
    }
    if (lane < k) {
        ids[(int64_t)m * ldid + lane] = id_lo;
        weights[(int64_t)m * ldwt + lane] = renormalize ? p_lo / total : p_lo;
    }
    if (32 + lane < k) {
        ids[(int64_t)m * ldid + 32 + lane] = id_hi;
        weights[(int64_t)m * ldwt + 32 + lane] = renormalize ? p_hi / total : p_hi;
    }
    griddep_launch_dependents();
}

}  // namespace

int router_topk_smem_bytes(int N) { return N * 5; }

cudaError_t launch_router_topk(const float *L, int64_t ldl, int M, int N, int k, int renormalize, float *weights,
                               int64_t ldwt, int32_t *ids, int64_t ldid, cudaStream_t stream, bool pdl) {
    if (M < 1 || N < 1 || N > kTopkMaxN || k < 1 || k > N || k > kTopkMaxK) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kTopkThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (N <= 1024) {
        // a warp per token, the row in registers
        cfg.gridDim = dim3((unsigned)((M + kTopkWarps - 1) / kTopkWarps), 1, 1);
        cfg.dynamicSmemBytes = 0;
        if (N <= 256)
            return cudaLaunchKernelEx(&cfg, router_topk_warp_kernel<8>, L, ldl, M, N, k, renormalize, weights, ldwt,
                                      ids, ldid);
        if (N <= 512)
            return cudaLaunchKernelEx(&cfg, router_topk_warp_kernel<16>, L, ldl, M, N, k, renormalize, weights, ldwt,
                                      ids, ldid);
        return cudaLaunchKernelEx(&cfg, router_topk_warp_kernel<32>, L, ldl, M, N, k, renormalize, weights, ldwt,
                                  ids, ldid);
    }
    cfg.gridDim = dim3((unsigned)M, 1, 1);
    cfg.dynamicSmemBytes = (size_t)router_topk_smem_bytes(N);
    return cudaLaunchKernelEx(&cfg, router_topk_kernel, L, ldl, N, k, renormalize, weights, ldwt, ids, ldid);
}

}  // namespace skinny
