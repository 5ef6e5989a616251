// tmem_gemm.cu -- the fifth-generation tensor-core backend: W and X tiles by
// tensor-map TMA, tcgen05.mma into tensor memory.
//
// Design source: "GLM-5.2 Blackwell decode optimizations", section
// "Implementation breakdown" item 3 (the decode projections qkv_a / q_b /
// eh_proj: the skinny GEMM at small M and a separate GEMM at medium M, picked
// per (N, K) by measured speed), and "[Perf][Feat] Add generic cuteDSL LL BF16
// router (GEMM)", item 2 (K split over the CTAs of a thread-block cluster,
// partial sums reduced through distributed shared memory).
//
// GB300 form.  A CTA owns TM = 128 or 64 rows of W (the MMA's M side; rows
// past N read as zeros) and, in a cluster of S CTAs along K, the K slice of
// its rank (KS elements, a whole number of ring stages).  The tokens are the
// MMA's N side (MT = 16, 32 or 64; rows past M read as zeros).  64-row tiles
// double the CTA count, which spreads a weight more evenly over the SMs.
//   * Thread 0 drives the TMA engine: per ring stage it loads stage_k / 64
//     boxes of W [TM rows x 64 K] and of X [MT rows x 64 K] through 2-D
//     tensor maps with the 128-byte swizzle (columns past K arrive as zeros),
//     all completing on the stage's "full" mbarrier.  W is a weight, so with
//     PDL the W boxes of the first ring pass are issued before
//     griddepcontrol.wait; X boxes only after it.
//   * Thread 32 issues tcgen05.mma kind::f16 (bf16 x bf16 -> fp32; M = TM,
//     N = MT, K = 16 each; operands from shared-memory descriptors, K-major,
//     128-byte swizzle) into an fp32 accumulator of MT columns in tensor
//     memory (M = 128: row r in lane r; M = 64: row 16w + i in lane 32w + i,
//     i < 16), frees each stage by tcgen05.commit on its "empty" mbarrier,
//     and signals "done" with a last commit.
//   * Warp 2 allocates the tensor-memory columns and frees them at the end.
//   * Epilogue, all four warps: warp w reads lanes 32w..32w+31 with
//     tcgen05.ld 32x32b: a thread holds one output column n, its registers
//     the tokens.  S = 1: Y is written directly (per token, a warp's columns
//     are one contiguous store).  S > 1: after one cluster barrier
//     (every CTA's MMAs are complete, so every ring is free) each CTA sends
//     the partials of rows owned by rank q = row / (TM / S) into q's ring
//     (slot = sending rank) with st.shared::cluster; after a second barrier
//     each owner adds slots 0..S-1 in that order and writes Y.  The MMA order
//     and the reduction order are fixed, so a plan's result is bit-identical
//     from run to run.
// Every mbarrier wait is bounded; a wait that gives up records an error in
// the device status word, the rest of the K loop is skipped, copies in flight
// are drained (bounded), and the CTA still takes part in both cluster
// barriers and frees its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace skinny {
namespace {

constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;
enum : int { kWaitDone = 5 };

// a box is `rows` x 64 bf16 (128 bytes per row)
__host__ __device__ constexpr int w_box_bytes(int TM) { return TM * 128; }
__host__ __device__ constexpr int x_box_bytes(int MT) { return MT * 128; }
__host__ __device__ constexpr int stage_bytes(int TM, int MT, int kb) { return kb * (w_box_bytes(TM) + x_box_bytes(MT)); }
__host__ __device__ constexpr int tmem_cols(int MT) { return MT <= 32 ? 32 : MT; }   // a power of two >= 32

// ------------------------------------------------------------------ TMA (tensor maps)
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// Box at (c0 = K element, c1 = row) of a 2-D tensor map into shared memory,
// completing on `bar`.  c0 is a multiple of 64 (128 bytes).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar) : "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(slot), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

// Shared-memory matrix descriptor: K-major operand in 128-byte swizzle atoms
// (8 rows x 128 bytes, rows 128 bytes apart, atoms 1024 bytes apart; the
// leading-dimension offset is not used by this layout).  `saddr` is the
// atom-aligned tile base plus 32 bytes per 16-element K step.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: fp32 D, bf16 A and B, both K-major,
// N = MT (bits 17-22, N / 8), M = TM (bits 24-28, M / 16).
template <int MT, int TM>
__host__ __device__ constexpr uint32_t idesc_bf16() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(MT >> 3) << 17) | ((uint32_t)(TM >> 4) << 24);
}
// D[tmem] (+)= A[smem] . B[smem]^T; accumulate = 0 overwrites D.
__device__ __forceinline__ void umma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}
// Arrive on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar)
                 : "memory");
}
// 16 consecutive fp32 columns of this thread's lane, waited for in the same
// statement so no use of the registers can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

struct TcParams {
    void *Y;
    int64_t ldy;
    int M, N, K;
    int KS;          // K elements per cluster rank, a multiple of 64 * kb
    int kb;          // 64-element boxes per ring stage
    int stages;
    int *status;
    uint64_t budget_ns;
    int out_bf16;
};

// Shared memory from the 1024-byte aligned base: the ring, then full[stages],
// empty[stages], done (8 bytes each), then the tensor-memory address.
__host__ __device__ inline int tc_layout_bytes(int TM, int MT, int kb, int stages) {
    return stages * stage_bytes(TM, MT, kb) + 8 * (2 * stages + 1) + 8;
}

template <int MT, int TM>
__global__ void __launch_bounds__(kTcThreads, 1)
tmem_gemm_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmx, const TcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;            // 128-byte swizzle atoms: 1024-byte aligned
    uint8_t *smem = smem_raw + (base - raw);
    constexpr int kWBox = w_box_bytes(TM);
    const int sbytes = stage_bytes(TM, MT, p.kb);
    const int stages = p.stages;
    const uint32_t bars = base + stages * sbytes;
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 8u * (stages + s); };
    const uint32_t done = bars + 16u * stages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + stages * sbytes + 8 * (2 * stages + 1));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = gridDim.x;
    const int rank = (S > 1) ? (int)cluster_ctarank() : 0;
    const int n0 = blockIdx.y * TM;
    const int kbeg = rank * p.KS;
    const int kend = min(p.K, kbeg + p.KS);
    const int sk = 64 * p.kb;
    const int nsteps = kend > kbeg ? (kend - kbeg + sk - 1) / sk : 0;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        mbar_init(done, 1);
        fence_mbarrier_init_cluster();
    }
    if (warp == 2) tmem_alloc(smem_u32(tmem_slot), tmem_cols(MT));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (tid == 0) {
        // ---- TMA producer (the other lanes of warp 0 wait for it at __syncwarp)
        prefetch_tensormap(&tmw);
        prefetch_tensormap(&tmx);
        const uint32_t tx = (uint32_t)sbytes;
        auto w_boxes = [&](int i, int s) {
            for (int b = 0; b < p.kb; ++b)
                tma_load_2d(base + s * sbytes + b * kWBox, &tmw, kbeg + (i * p.kb + b) * 64, n0, full(s));
        };
        auto x_boxes = [&](int i, int s) {
            for (int b = 0; b < p.kb; ++b)
                tma_load_2d(base + s * sbytes + p.kb * kWBox + b * x_box_bytes(MT), &tmx,
                            kbeg + (i * p.kb + b) * 64, 0, full(s));
        };
        const int pre = min(nsteps, stages);
        for (int i = 0; i < pre; ++i) {
            mbar_arrive_expect_tx(full(i), tx);
            w_boxes(i, i);                       // the weight: before the PDL wait
        }
        griddep_wait();
        griddep_launch_dependents();
        for (int i = 0; i < pre; ++i) x_boxes(i, i);
        int issued = pre;
        for (int i = pre; i < nsteps; ++i) {
            const int s = i % stages;
            if (!mbar_wait_bounded(empty(s), (uint32_t)((i / stages - 1) & 1), p.budget_ns)) {
                report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitProducerEmpty);
                break;
            }
            mbar_arrive_expect_tx(full(s), tx);
            w_boxes(i, s);
            x_boxes(i, s);
            issued = i + 1;
        }
        // every copy issued has landed before the ring is reused or the CTA exits
        for (int i = max(0, issued - stages); i < issued; ++i)
            if (!mbar_wait_bounded(full(i % stages), (uint32_t)((i / stages) & 1), kDrainNs))
                report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitDrain);
    } else if (tid == 32) {
        // ---- MMA issuer
        griddep_wait();
        griddep_launch_dependents();
        constexpr uint32_t idesc = idesc_bf16<MT, TM>();
        for (int i = 0; i < nsteps; ++i) {
            const int s = i % stages;
            if (!mbar_wait_bounded(full(s), (uint32_t)((i / stages) & 1), p.budget_ns)) {
                report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitConsumerFull);
                break;
            }
            tc_fence_after();
            const uint32_t wst = base + s * sbytes;
            const uint32_t xst = wst + p.kb * kWBox;
            for (int b = 0; b < p.kb; ++b)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    umma_bf16(tmem, sw128_desc(wst + b * kWBox + 32 * j), sw128_desc(xst + b * x_box_bytes(MT) + 32 * j),
                              idesc, (i | b | j) != 0 ? 1u : 0u);
            umma_commit(empty(s));               // the stage is free once these MMAs have read it
        }
        umma_commit(done);                       // also when the loop gave up: tracks what was issued
    } else {
        griddep_wait();                          // Y may be read or written by the preceding kernel
        griddep_launch_dependents();
    }
    __syncwarp();

    // ---- epilogue: accumulator rows 32*warp + lane, columns = tokens
    if (!mbar_wait_bounded(done, 0, p.budget_ns)) {
        if (lane == 0) report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitDone);
        if (!mbar_wait_bounded(done, 0, kDrainNs) && lane == 0)
            report_status(p.status, SKINNY_ERR_DEVICE_TIMEOUT, kWaitDrain);
    }
    tc_fence_after();
    const int M = p.M;
    float v[MT];
#pragma unroll
    for (int c = 0; c < MT / 16; ++c) {
        if (16 * c < M && nsteps > 0) {          // warp-uniform
            tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + 16 * c, v + 16 * c);
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[16 * c + j] = 0.f;
        }
    }
    if (nsteps == 0) {
#pragma unroll
        for (int j = 0; j < MT; ++j) v[j] = 0.f;   // an empty K slice adds nothing
    }
    // accumulator row of this thread (M = 64: lanes 16..31 of each warp hold none)
    const int row = (TM == 128) ? 32 * warp + lane : 16 * warp + lane;
    const bool has_row = (TM == 128) || lane < 16;
    if (S == 1) {
        const int n = n0 + row;
        if (has_row && n < p.N) {
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (m < M) store_y(p.Y, p.out_bf16, m * p.ldy + n, v[m]);
        }
    } else {
        const int R = TM / S;                    // rows owned by each rank
        cluster_arrive_release();                // every CTA of the cluster is past its MMAs
        cluster_wait_acquire();
        if (has_row) {
            const int q = row / R, rl = row - q * R;
            const uint32_t dst = mapa_shared(base, (uint32_t)q);
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (m < M) st_shared_cluster_f32(dst + 4u * (uint32_t)((rank * M + m) * R + rl), v[m]);
        }
        cluster_arrive_release();                // every partial is in its owner's slots
        cluster_wait_acquire();
        const float *slots = reinterpret_cast<const float *>(smem);
        for (int i = tid; i < M * R; i += kTcThreads) {
            const int m = i / R, r = i - m * R;
            const int n = n0 + rank * R + r;
            float acc = slots[m * R + r];
            for (int src = 1; src < S; ++src) acc += slots[(src * M + m) * R + r];
            if (n < p.N) store_y(p.Y, p.out_bf16, m * p.ldy + n, acc);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols(MT));
    }
}

using TcKernel = void (*)(const CUtensorMap, const CUtensorMap, const TcParams);
const TcKernel kTc[3][2] = {{&tmem_gemm_kernel<16, 128>, &tmem_gemm_kernel<16, 64>},
                            {&tmem_gemm_kernel<32, 128>, &tmem_gemm_kernel<32, 64>},
                            {&tmem_gemm_kernel<64, 128>, &tmem_gemm_kernel<64, 64>}};

int tc_index(int M) { return M <= 16 ? 0 : M <= 32 ? 1 : 2; }

// The driver's tensor-map encoder, resolved once through the runtime (no link
// against the driver library).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// bf16 [rows, cols] with row stride ld (elements), boxes of 64 columns x box_rows
// rows, 128-byte swizzle, zeros outside the tensor.
bool encode_bf16_2d(CUtensorMap *map, const void *ptr, int cols, int rows, int64_t ld, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int tc_tokens(int M) { return 16 << tc_index(M); }

bool tc_supported(int M) { return M >= 1 && M <= SKINNY_MAX_M; }

int tc_smem_bytes(int M, int block_n, int stage_k, int stages, int split_k) {
    const int MT = tc_tokens(M);
    const int kb = stage_k / 64;
    int bytes = tc_layout_bytes(block_n, MT, kb, stages);
    // S > 1: the ring also receives the partials (S slots of M x block_n / S fp32)
    if (split_k > 1 && stages * stage_bytes(block_n, MT, kb) < block_n * M * 4) return 1 << 30;
    // at most 7 resident CTAs per SM, so their tensor memory (<= 64 columns
    // each) always fits in the SM's 512 columns and an allocation never waits
    if (bytes < kTcMinSmem - 1024) bytes = kTcMinSmem - 1024;
    return bytes + 1024;                         // slack for the 1024-byte alignment
}

cudaError_t tc_prepare() {
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 2; ++j) {
            cudaError_t e = set_max_dyn_smem(kTc[i][j]);
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

cudaError_t launch_tc(const GemmArgs &a, const skinny_plan_t &pl, const LaunchCtx &c) {
    const int S = pl.split_k;
    const int TM = pl.block_n;
    if (!tc_supported(a.M) || (TM != 128 && TM != 64) || S < 1 || S > kSplitMaxCluster || (TM % S) != 0 ||
        pl.stage_k < 64 || pl.stage_k > kTcMaxBK || pl.stage_k % 64 || pl.stages < 1 ||
        pl.stages > kSplitMaxStages || pl.k_chunk % pl.stage_k || (int64_t)pl.k_chunk * S < a.K ||
        pl.grid_x != S || pl.grid_y != (a.N + TM - 1) / TM || pl.smem_bytes < kTcMinSmem ||
        pl.smem_bytes < tc_smem_bytes(a.M, TM, pl.stage_k, pl.stages, S))
        return cudaErrorInvalidValue;
    if ((reinterpret_cast<uintptr_t>(a.X) & 15) || (a.ldx & 7) || (reinterpret_cast<uintptr_t>(a.W) & 15) ||
        (a.ldw & 7))
        return cudaErrorInvalidValue;
    const int idx = tc_index(a.M);
    CUtensorMap tmw, tmx;
    if (!encode_bf16_2d(&tmw, a.W, a.K, a.N, a.ldw, TM) || !encode_bf16_2d(&tmx, a.X, a.K, a.M, a.ldx, 16 << idx))
        return cudaErrorInvalidValue;
    TcParams p;
    p.Y = a.Y;
    p.ldy = a.ldy;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.KS = pl.k_chunk;
    p.kb = pl.stage_k / 64;
    p.stages = pl.stages;
    p.status = c.status;
    p.budget_ns = c.budget_ns;
    p.out_bf16 = a.out_bf16;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, pl.grid_y, 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem_bytes;
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
    return cudaLaunchKernelEx(&cfg, kTc[idx][TM == 128 ? 0 : 1], tmw, tmx, p);
}

}  // namespace skinny
