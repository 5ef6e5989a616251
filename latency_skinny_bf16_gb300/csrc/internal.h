// internal.h -- host-side declarations shared by the translation units of
// libskinny_gemm.so.  Nothing here is part of the public C ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "skinny_gemm.h"

namespace skinny {

// Token counts: every kernel takes M <= 16; the cluster split-K kernel with
// the MMA consumer also takes 17..64 (the SKINNY_MAX_M of the C ABI).
constexpr int kMaxMSmall = 16;
constexpr int kMaxMSplitMma = SKINNY_MAX_M;
int splitk_mma_tokens(int M);   // MMA token bucket: 8, 16, 32 or 64

struct GemmArgs {
    const uint16_t *X;
    int64_t ldx;
    const uint16_t *W;
    int64_t ldw;
    void *Y;             // fp32, or bf16 bits when out_bf16
    int64_t ldy;
    int M, N, K;
    int out_bf16;
};

struct LaunchCtx {
    cudaStream_t stream;
    bool pdl;            // programmatic dependent launch attribute
    // When this kernel lets the next launch start (griddepcontrol.launch_dependents):
    // false = at once (short calls: the next call's prologue overlaps all of this
    // one); true = once each CTA has issued its last weight load (long,
    // bandwidth-bound calls: the next call's CTAs fill the SMs this one leaves,
    // and do not take bandwidth or slots from its main loop).
    bool late;
    int *status;         // device status word (error reports from bounded waits)
    uint64_t budget_ns;  // budget of each bounded wait; 0 = give up at once (test hook)
};

// ---- dot-product backend (dotprod.cu)
constexpr int kDotThreads = 128;
int dotprod_smem_bytes(int M, int block_n, int k_chunk);
bool dotprod_supported(int M, int vec_elems, int block_n);
cudaError_t dotprod_prepare();   // per-device kernel attributes
cudaError_t launch_dotprod(const GemmArgs &a, const skinny_plan_t &p, const LaunchCtx &c);

// ---- dot-product backend with mma.sync arithmetic (dotmma.cu): block_n 16/32/64
int dotmma_smem_bytes(int M, int block_n, int k_chunk, int split_k);
__host__ __device__ int dotmma_k_slice(int K, int S);   // K elements per cluster rank
bool dotmma_split_ok(int M, int K, int S);              // S == 1, or a cluster split K can take
bool dotmma_supported(int M, int block_n);
int dotmma_tokens(int M);   // token bucket of the instantiation: 8, 16, 32 or 64
cudaError_t dotmma_prepare();
cudaError_t launch_dotmma(const GemmArgs &a, const skinny_plan_t &p, const LaunchCtx &c);

// ---- cluster split-K backend (splitk.cu)
// Consumer warps per split-K CTA.  The FMA consumer maps 4 warps x 4 rows onto
// the 16-row tile.  The MMA consumer splits each stage's 16-wide K steps over
// its warps: 8 when a stage holds at least 1024 K elements and the token
// bucket is at most 16 (measured on GB300: 5-6% faster there; shorter stages
// lose to the larger reduction, 32 / 64 tokens to the larger partial buffers),
// else 4.
constexpr int kSplitConsumerWarps = 4;
constexpr int kSplitMmaWarps = 8;
__host__ __device__ constexpr int splitk_consumer_warps(int consumer, int mt, int stage_k) {
    return (consumer == SKINNY_CONSUMER_MMA && mt <= 16 && stage_k >= 1024) ? kSplitMmaWarps
                                                                            : kSplitConsumerWarps;
}
__host__ __device__ constexpr int splitk_threads(int consumer, int mt, int stage_k) {
    return (splitk_consumer_warps(consumer, mt, stage_k) + 1) * 32;   // + one producer warp
}
constexpr int kSplitThreads = (kSplitConsumerWarps + 1) * 32;
constexpr int kSplitBK = 256;        // default K elements per ring stage (one-shot slices)
constexpr int kSplitStreamBK = 1024; // K elements per ring stage when streaming (2 KB per W row)
constexpr int kSplitMaxBK = 2048;
constexpr int kSplitMaxCluster = 8;
constexpr int kSplitMaxStages = 16;
int splitk_smem_bytes(int M, int consumer, int block_n, int stages, int k_slice, int split_k, int stage_k);
bool splitk_supported(int M, int consumer, int block_n);
cudaError_t splitk_prepare();
cudaError_t launch_splitk(const GemmArgs &a, const skinny_plan_t &p, const LaunchCtx &c);

// ---- K-outer streaming backend (stream.cu): one CTA per SM, whole K per
// 16-row tile, X streamed through the ring chunk by chunk
constexpr int kStreamMaxTiles = 4;   // 16-row tiles per CTA (register accumulators)
int stream_smem_bytes(int M, int stages, int stage_k);
bool stream_supported(int M);
cudaError_t stream_prepare();
cudaError_t launch_stream(const GemmArgs &a, const skinny_plan_t &p, const LaunchCtx &c);

// ---- fifth-generation tensor-core backend (tmem_gemm.cu): W rows split into
// C balanced ranges of 8-row groups (clusters of split_k CTAs along K), tiles of
// at most 128 rows on the MMA's M side (block_n = 64 or 128), tokens on its N
// side (16 / 32 / 64), W and X boxes by tensor-map TMA, the tensor-memory
// accumulator drained into fp32 registers after every ring stage
constexpr int kTcThreads = 192;        // producer warp, MMA warp, four draining warps
constexpr int kTcMaxBK = 256;          // K elements per ring stage: 64..256, multiple of 64 (<= 16 MMAs)
constexpr int kTcCtasPerSm = 2;        // the default grid: two CTAs per SM
constexpr int kTcSmemBudget = 110 * 1024;   // per CTA, so two fit in an SM's 228 KB
// Shared memory asked for at least, so an SM holds at most two CTAs and their
// tensor memory (256 columns each) never exceeds its 512 columns
constexpr int kTcMinSmem = 77 * 1024;
int tc_tokens(int M);                  // MMA N of the instantiation: 16, 32 or 64
bool tc_supported(int M);
int tc_smem_bytes(int M, int N, int K, int block_n, int stage_k, int stages, int split_k, int clusters, bool norm);
// The plan for (M, N, K); zero arguments take the default.  false if none fits.
bool tc_make_plan(int M, int N, int K, int force_bn, int force_s, int force_stages, int force_bk, int force_c,
                  int num_sms, skinny_plan_t *p);
// The fused query RMS norm in front of the GEMM (X = rms_norm(xr) * gamma,
// also stored to xn): the tcgen05 plan `gemm` with the ring shortened so the
// rank's whole K slice of X fits beside it.  Up to kTcNormMaxM tokens.
constexpr int kTcNormMaxM = 16;
struct TcNormArgs {
    const uint16_t *xr;
    int64_t ldxr;
    const uint16_t *gamma;
    float eps;
    uint16_t *xn;
    int64_t ldxn;
};
bool tc_make_norm_plan(int M, int N, int K, const skinny_plan_t &gemm, skinny_plan_t *p);
cudaError_t tc_prepare();
cudaError_t launch_tc(const GemmArgs &a, const skinny_plan_t &p, const LaunchCtx &c,
                      const TcNormArgs *norm = nullptr);

// ---- dot-product backend for fp32 weights (dotprod_f32w.cu): vec_elems 4/2/1 fp32, block_n 1/2/4
bool dotprod_f32w_supported(int M, int vec_elems, int block_n);
int dotprod_f32w_smem_bytes(int M, int block_n, int k_chunk);
cudaError_t dotprod_f32w_prepare();
cudaError_t launch_dotprod_f32w(const uint16_t *X, int64_t ldx, const float *W, int64_t ldw, float *Y, int64_t ldy,
                                int M, int N, int K, const skinny_plan_t &p, const LaunchCtx &c);

// ---- query RMS norm in front of the q_b projection (rmsnorm.cu)
cudaError_t launch_rmsnorm(const uint16_t *X, int64_t ldx, const uint16_t *G, float eps, int M, int K, uint16_t *XN,
                           int64_t ldxn, cudaStream_t stream, bool pdl);

// ---- router epilogue (topk.cu): softmax + top-k over each token's logits
constexpr int kTopkMaxN = 8192;   // logits per token (shared memory: 5 bytes each)
constexpr int kTopkMaxK = 64;
int router_topk_smem_bytes(int N);
cudaError_t launch_router_topk(const float *L, int64_t ldl, int M, int N, int k, int renormalize, float *weights,
                               int64_t ldwt, int32_t *ids, int64_t ldid, cudaStream_t stream, bool pdl);

// Per-CTA dynamic shared memory the dispatcher may plan for (GB300: 232448
// bytes opt-in per block, less a margin for the kernels' static shared memory).
constexpr int kMaxDynSmem = 227 * 1024 - 1024;

// Allow `fn` the device's opt-in shared memory per block, less its static part.
template <typename F>
inline cudaError_t set_max_dyn_smem(F *fn) {
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void *>(fn));
    if (e != cudaSuccess) return e;
    const int limit = optin - (int)fa.sharedSizeBytes;
    return cudaFuncSetAttribute(reinterpret_cast<const void *>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                limit < kMaxDynSmem ? limit : kMaxDynSmem);
}

}  // namespace skinny
