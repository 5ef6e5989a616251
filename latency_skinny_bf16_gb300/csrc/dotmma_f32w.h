// dotmma_f32w.h -- the tensor-core dot-product for fp32 weights (dotmma_f32w.cu).
// W rows 16-byte aligned (W and ldw), K % 32 == 0, M <= 16; block_n 16 or 32;
// split_k = S CTAs of a cluster along K (1..8, every rank given some K).
#pragma once
#include "internal.h"

namespace skinny {

__host__ __device__ int dotmma_f32w_k_slice(int K, int S);   // K elements per cluster rank
bool dotmma_f32w_split_ok(int K, int S);
bool dotmma_f32w_supported(int M, int block_n);
int dotmma_f32w_threads(int M);   // threads per CTA: 256 up to 8 tokens, 128 above
int dotmma_f32w_smem_bytes(int M, int block_n, int K, int split_k);
cudaError_t dotmma_f32w_prepare();
cudaError_t launch_dotmma_f32w(const uint16_t *X, int64_t ldx, const float *W, int64_t ldw, float *Y, int64_t ldy,
                               int M, int N, int K, const skinny_plan_t &p, const LaunchCtx &c);

}  // namespace skinny
