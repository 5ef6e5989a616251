// api.cu -- the C ABI of libskinny_gemm.so: argument checks, per-device set-up,
// the (M, K, N) dispatcher with its measured tuning table, options, and the
// device status word.
//
// Dispatch follows "[Perf][Feat] Add generic cuteDSL LL BF16 router (GEMM)",
// section "Key source snippets" (ll_bf16.py: LLBf16Gemm.dispatch picks the
// dot-product kernel when M is at most a per-(K, N) tuned maximum or K < 2048,
// otherwise split-K with a per-(K, N, M) tuned (split_k, num_stages)), and the
// review notes there (bf16-only, M <= 16, no over-strong alignment
// assumption).  Here the tuning table is measured on GB300 and compiled in, and
// every plan is checked against what the kernels support before launch.
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cmath>
#include <cstring>
#include <mutex>
#include <set>
#include <tuple>

#include "internal.h"
#include "dotmma_f32w.h"

namespace skinny {
namespace {

// ------------------------------------------------------------------ device status word
__device__ int g_status_word;
__device__ int g_status_taken;   // the value the last read-and-clear took

// Read and clear the status word in one atomic step, so a report that lands
// at any moment is either returned now or kept for the next read.
__global__ void status_take_kernel() { g_status_taken = atomicExch(&g_status_word, 0); }
std::mutex g_status_mu;          // one reader of g_status_taken at a time

// K == 0: Y is the empty sum, +0 (fp32 or bf16 bits).
__global__ void zero_fill_kernel(void *Y, int64_t ldy, int M, int N, int out_bf16) {
    const int64_t total = (int64_t)M * N;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / N, n = i - m * N;
        if (out_bf16) static_cast<uint16_t *>(Y)[m * ldy + n] = 0;
        else static_cast<float *>(Y)[m * ldy + n] = 0.f;
    }
}

// ------------------------------------------------------------------ options
std::atomic<int> g_opt_pdl{-1};            // -1: not yet read from the environment
std::atomic<int> g_opt_force_backend{0};
std::atomic<int> g_opt_force_consumer{0};
std::atomic<int> g_opt_force_split_k{0};
std::atomic<int> g_opt_force_block_n{0};
std::atomic<int> g_opt_force_stages{0};
std::atomic<int> g_opt_wait_us{500000};
std::atomic<int> g_opt_force_grid_y{0};
std::atomic<int> g_opt_force_stage_k{0};
std::atomic<int> g_opt_log{-1};
std::atomic<int> g_opt_fuse_norm{0};   // the fused q_b norm measured slower than two launches
std::atomic<int> g_opt_late_trigger{0};

int env_flag(const char *name) {
    const char *v = std::getenv(name);
    return (v && v[0] && std::strcmp(v, "0") != 0) ? 1 : 0;
}
int opt_pdl() {
    int v = g_opt_pdl.load();
    if (v < 0) {
        const char *e = std::getenv("SKINNY_PDL");
        v = (e && std::strcmp(e, "2") == 0) ? 2 : env_flag("SKINNY_PDL");
        g_opt_pdl.store(v);
    }
    return v;
}
// Programmatic dependent launch for a call moving `w_bytes` of weight, W
// staged through shared memory by the copy engine (`w_by_tma`: split-K,
// K-outer streaming, tcgen05) or loaded into registers (the dot-product
// kernels).  Mode 1 gives it to every call of the first kind and to calls of
// the second kind under kPdlMaxWBytes.  A load into registers passes through
// the SM's L1, whose share of the SM's on-chip memory is what the kernels
// resident on the SM leave of it: a dot-product CTA that starts early on an SM
// still holding a shared-memory-heavy predecessor (split-K, tcgen05) runs with
// that small L1, which caps its loads in flight.  Measured on GB300: the
// 24576 x 1536 dot-product call took 14.5 us after such a predecessor without
// PDL and about 36 us with it (the same call with the largest shared-memory
// carveout, no PDL: 30 us), while a chain of the same call gained nothing from
// PDL.  Calls whose W goes through shared memory do not depend on L1 and gain:
// the decode step of the projection weights went from 317 to 306 us, chains
// of one projection call by 0.6-2.5 us per call, a chain of 64 router calls
// from 285 to 164 us.
constexpr double kPdlMaxWBytes = 16e6;
int pdl_for(double w_bytes, bool w_by_tma) {
    const int v = opt_pdl();
    return (v == 2 || (v == 1 && (w_by_tma || w_bytes < kPdlMaxWBytes))) ? 1 : 0;
}

// With SKINNY_OPT_LATE_TRIGGER, weights of 16 MB and more let the next launch
// start late (see LaunchCtx::late).  Off by default: with PDL given to the
// plans that stage W through shared memory only, the decode step of the
// projection weights measured 296 us with the trigger at kernel entry against
// 302 us with the late one on GB300.
bool late_trigger(double w_bytes) { return g_opt_late_trigger.load() != 0 && w_bytes >= 16e6; }
int opt_log() {
    int v = g_opt_log.load();
    if (v < 0) { v = env_flag("SKINNY_LOG"); g_opt_log.store(v); }
    return v;
}

// ------------------------------------------------------------------ per-device state
constexpr int kMaxDevices = 64;
struct DeviceState {
    std::once_flag once;
    skinny_status_t status = SKINNY_ERR_NO_DEVICE;
    int num_sms = 0;
    int *status_word = nullptr;
};
DeviceState g_dev[kMaxDevices];

skinny_status_t init_device_current(DeviceState &d, int device) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return SKINNY_ERR_NO_DEVICE;
    if (major != 10 || minor != 3) return SKINNY_ERR_NO_DEVICE;   // built for sm_103a only
    if (dotprod_prepare() != cudaSuccess || dotmma_prepare() != cudaSuccess || splitk_prepare() != cudaSuccess ||
        stream_prepare() != cudaSuccess || dotprod_f32w_prepare() != cudaSuccess ||
        dotmma_f32w_prepare() != cudaSuccess || tc_prepare() != cudaSuccess)
        return SKINNY_ERR_LAUNCH;
    void *sym = nullptr;
    if (cudaGetSymbolAddress(&sym, g_status_word) != cudaSuccess) return SKINNY_ERR_LAUNCH;
    d.num_sms = sms;
    d.status_word = static_cast<int *>(sym);
    return SKINNY_OK;
}

// Runs the set-up once per device, with that device current.
skinny_status_t ensure_device(int device) {
    if (device < 0 || device >= kMaxDevices) return SKINNY_ERR_NO_DEVICE;
    DeviceState &d = g_dev[device];
    std::call_once(d.once, [&] {
        int prev = -1;
        if (cudaGetDevice(&prev) != cudaSuccess) { d.status = SKINNY_ERR_NO_DEVICE; return; }
        if (prev != device && cudaSetDevice(device) != cudaSuccess) { d.status = SKINNY_ERR_NO_DEVICE; return; }
        d.status = init_device_current(d, device);
        if (prev != device) cudaSetDevice(prev);
    });
    return d.status;
}

skinny_status_t current_device(int *device) {
    if (cudaGetDevice(device) != cudaSuccess) return SKINNY_ERR_NO_DEVICE;
    return ensure_device(*device);
}

// ------------------------------------------------------------------ argument checks
bool ranges_overlap(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

// Host-only validation; no CUDA call.  *noop is set when there is nothing to launch.
// y_bytes: size of one Y element (4 for fp32, 2 for bf16).
skinny_status_t validate(const uint16_t *X, int ldx, const void *W, int ldw, const void *Y, int ldy,
                         int M, int N, int K, bool *noop, int y_bytes = 4, int w_bytes = 2) {
    *noop = false;
    if (M < 0 || N < 0 || K < 0) return SKINNY_ERR_INVALID_VALUE;
    if (M > SKINNY_MAX_M) return SKINNY_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) { *noop = true; return SKINNY_OK; }
    if (Y == nullptr || ldy < N) return SKINNY_ERR_INVALID_VALUE;
    if (reinterpret_cast<uintptr_t>(Y) & (uintptr_t)(y_bytes - 1)) return SKINNY_ERR_MISALIGNED;
    if (K == 0) return SKINNY_OK;
    if (X == nullptr || W == nullptr || ldx < K || ldw < K) return SKINNY_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(X) & 1) || (reinterpret_cast<uintptr_t>(W) & (uintptr_t)(w_bytes - 1)))
        return SKINNY_ERR_MISALIGNED;
    const uintptr_t y0 = reinterpret_cast<uintptr_t>(Y);
    const uintptr_t y1 = y0 + (uintptr_t)(((int64_t)(M - 1) * ldy + N) * y_bytes);
    const uintptr_t x0 = reinterpret_cast<uintptr_t>(X);
    const uintptr_t x1 = x0 + (uintptr_t)(((int64_t)(M - 1) * ldx + K) * 2);
    const uintptr_t w0 = reinterpret_cast<uintptr_t>(W);
    const uintptr_t w1 = w0 + (uintptr_t)(((int64_t)(N - 1) * ldw + K) * w_bytes);
    if (ranges_overlap(y0, y1, x0, x1) || ranges_overlap(y0, y1, w0, w1)) return SKINNY_ERR_INVALID_VALUE;
    return SKINNY_OK;
}

// ------------------------------------------------------------------ dispatcher
struct TunedEntry {
    int K, N, m_lo, m_hi;
    int backend, consumer, split_k, block_n, stages, stage_k, clusters;
};
const TunedEntry kTuned[] = {
#include "tuning_table.inc"
    {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0}};

const TunedEntry *lookup_tuned(int M, int N, int K) {
    for (const TunedEntry &e : kTuned)
        if (e.K == K && e.N == N && M >= e.m_lo && M <= e.m_hi) return &e;
    return nullptr;
}

int widest_vec(const uint16_t *W, int ldw) {
    const uintptr_t w = reinterpret_cast<uintptr_t>(W);
    if ((w & 15) == 0 && (ldw & 7) == 0) return 8;
    if ((w & 7) == 0 && (ldw & 3) == 0) return 4;
    if ((w & 3) == 0 && (ldw & 1) == 0) return 2;
    return 1;
}

int pow2_floor(int v) { int p = 1; while (p * 2 <= v) p *= 2; return p; }

constexpr int kDotXBudget = 96 * 1024;     // X bytes staged per dot-product CTA
constexpr int kSplitXBudget = 160 * 1024;  // X slice bytes per split-K CTA
constexpr int kMmaXBudget = 64 * 1024;     // X bytes staged per tensor-core dot-product CTA (3 CTAs / SM)

bool plan_dotprod(int M, int N, int K, int vec, int force_bn, int num_sms, skinny_plan_t *p) {
    int bn = force_bn;
    if (bn == 0) {
        bn = (vec == 8) ? pow2_floor(N / (2 * num_sms) > 0 ? N / (2 * num_sms) : 1) : 1;
        if (bn > 8) bn = 8;
    }
    if (!dotprod_supported(M, vec, bn)) return false;
    // Whole K when it fits; otherwise chunks of a multiple of 8 * 128 elements,
    // so every K vector lands on the same thread whatever M is (each thread's
    // summation order, hence the result, is independent of M and of chunking).
    const int k8 = (K + 7) & ~7;
    int kc = (kDotXBudget / (2 * M)) & ~7;
    if (kc >= k8) {
        kc = k8;
    } else {
        kc = (kc / (8 * kDotThreads)) * (8 * kDotThreads);
        if (kc < 8 * kDotThreads) kc = 8 * kDotThreads;
    }
    p->backend = SKINNY_BACKEND_DOTPROD;
    p->consumer = SKINNY_CONSUMER_FMA;
    p->vec_elems = vec;
    p->block_n = bn;
    p->split_k = 1;
    p->stages = 0;
    p->k_chunk = kc;
    p->grid_x = (N + bn - 1) / bn;
    p->grid_y = 1;
    p->threads = kDotThreads;
    p->smem_bytes = dotprod_smem_bytes(M, bn, kc);
    return p->smem_bytes <= kMaxDynSmem;
}

// Dot-product layout with mma.sync arithmetic: block_n = 16 * row tiles;
// split_k > 1 cuts K over the CTAs of a cluster (grid split_k x blocks).
bool plan_dotmma(int M, int N, int K, int vec, int force_bn, int force_s, int num_sms, skinny_plan_t *p) {
    if (vec != 8 || K % 32 != 0 || K < 32) return false;
    const int S = force_s > 0 ? force_s : 1;
    if (!dotmma_split_ok(M, K, S)) return false;
    int bn = force_bn;
    if (bn == 0) {
        // enough CTAs for every SM, fewer X re-reads when N is large
        bn = 16;
        while (bn < 64 && (int64_t)S * ((N + 2 * bn - 1) / (2 * bn)) >= 2 * num_sms) bn *= 2;
    }
    if (!dotmma_supported(M, bn)) return false;
    const int MT = dotmma_tokens(M);
    const int KS = S > 1 ? dotmma_k_slice(K, S) : K;
    // 8 / 16 tokens: 64 KB of X per CTA (3 CTAs per SM); 32 / 64: 96 KB, so
    // the chunks stay at least 768 elements long
    int kc = ((MT >= 32 ? 96 * 1024 : kMmaXBudget) / (2 * MT)) & ~31;
    if (kc >= KS) kc = KS;
    if (kc < 32) kc = 32;
    const int blocks = (N + bn - 1) / bn;
    p->backend = SKINNY_BACKEND_DOTPROD;
    p->consumer = SKINNY_CONSUMER_MMA;
    p->vec_elems = 8;
    p->block_n = bn;
    p->split_k = S;
    p->stages = 0;
    p->stage_k = 0;
    p->k_chunk = kc;
    p->grid_x = S > 1 ? S : blocks;
    p->grid_y = S > 1 ? blocks : 1;
    if (p->grid_y > 65535) return false;
    p->threads = kDotThreads;
    p->smem_bytes = dotmma_smem_bytes(M, bn, kc, S);
    return p->smem_bytes <= kMaxDynSmem;
}

bool plan_splitk(int M, int N, int K, int vec, int consumer, int force_s, int force_stages, int force_c,
                 int force_bk, int num_sms, skinny_plan_t *p) {
    if (vec != 8 || K % 8 != 0 || K < 8) return false;
    if (consumer == SKINNY_CONSUMER_MMA && K % 16 != 0) return false;
    if (!splitk_supported(M, consumer, 16)) return false;
    const int tiles = (N + 15) / 16;
    int S = force_s;
    if (S == 0) {
        S = num_sms / tiles;
        const int max_by_k = (K + kSplitBK - 1) / kSplitBK;
        if (S > max_by_k) S = max_by_k;
        if (S > kSplitMaxCluster) S = kSplitMaxCluster;
        if (S < 1) S = 1;
    }
    if (S < 1 || S > kSplitMaxCluster) return false;
    for (;; ++S) {
        if (S > kSplitMaxCluster) return false;
        const int ks = ((K + S - 1) / S + 15) & ~15;
        const int xbytes = M * (((ks * 2 + 127) & ~127) + 16);   // the M token rows of X
        if (xbytes > kSplitXBudget && !force_s) continue;
        // Ring chunk: each W row of a chunk is one bulk copy, and the copy
        // engine's cost is per copy (~50 ns each on GB300, measured), so
        // chunks are as long as possible: the whole slice (up to 2048 elements,
        // 4 KB per row) in one stage when a cluster owns a single tile (one
        // shot: every W byte requested at kernel start), and up to 2048-element
        // chunks when persistent clusters stream many tiles.
        int bk = force_bk ? force_bk : ((ks + 63) / 64) * 64;
        if (!force_bk && bk > kSplitMaxBK) bk = kSplitMaxBK;
        if (bk < 64 || bk > kSplitMaxBK || bk % 64) return false;
        int stages = 0;
        for (;;) {
            // one shot when the slice is at most 8 chunks, else the deepest ring
            // that fits; if even 2 stages do not fit, halve the chunk
            const int nchunks = (ks + bk - 1) / bk;
            stages = force_stages ? force_stages : (nchunks <= 8 ? (nchunks < 1 ? 1 : nchunks) : kSplitMaxStages);
            while (!force_stages && stages > 2 && splitk_smem_bytes(M, consumer, 16, stages, ks, S, bk) > kMaxDynSmem)
                --stages;
            if (splitk_smem_bytes(M, consumer, 16, stages, ks, S, bk) <= kMaxDynSmem) break;
            if (force_bk || bk <= kSplitBK) break;
            bk = ((bk / 2 + 63) / 64) * 64;
        }
        if (stages < 1 || stages > kSplitMaxStages) return false;
        const int smem = splitk_smem_bytes(M, consumer, 16, stages, ks, S, bk);
        if (smem > kMaxDynSmem) return false;
        // Persistent clusters: as many as can be resident (shared memory, and
        // at most 3 CTAs of 160 threads per SM by registers), with the tiles
        // spread evenly over them.
        int per_sm = (228 * 1024) / (smem + 1024);
        if (per_sm > 3) per_sm = 3;
        if (per_sm < 1) per_sm = 1;
        int cap = num_sms * per_sm / S;
        if (cap < 1) cap = 1;
        // 32 / 64 tokens keep one partial-sum buffer: one tile per cluster
        const bool one_tile = S > 1 && consumer == SKINNY_CONSUMER_MMA && splitk_mma_tokens(M) >= 32;
        if (one_tile && force_c && force_c < tiles) return false;
        int C = force_c;
        if (one_tile) {
            C = tiles;
        } else if (C == 0) {
            if (tiles <= cap) {
                C = tiles;
            } else {
                const int per = (tiles + cap - 1) / cap;
                C = (tiles + per - 1) / per;
            }
        }
        if (C < 1 || C > 65535) return false;
        if (C > tiles) C = tiles;
        p->backend = SKINNY_BACKEND_SPLITK;
        p->consumer = consumer;
        p->vec_elems = 8;
        p->block_n = 16;
        p->split_k = S;
        p->stages = stages;
        p->stage_k = bk;
        p->k_chunk = ks;
        p->grid_x = S;
        p->grid_y = C;
        p->threads = splitk_threads(consumer, consumer == SKINNY_CONSUMER_MMA ? splitk_mma_tokens(M) : M, bk);
        p->smem_bytes = smem;
        return true;
    }
}

// K-outer streaming plan: one CTA per SM (at most kStreamMaxTiles tiles
// each), the longest chunks up to 2048 elements that split K evenly, and the
// deepest ring that fits (at least one chunk's X and W entries, plus one).
bool plan_stream(int M, int N, int K, int vec, bool x_ok, int force_c, int force_stages, int force_bk,
                 int num_sms, skinny_plan_t *p) {
    if (vec != 8 || !x_ok || K % 16 != 0 || K < 16 || !stream_supported(M)) return false;
    const int tiles = (N + 15) / 16;
    int C = force_c ? force_c : (tiles < num_sms ? tiles : num_sms);
    if (C > tiles) C = tiles;
    if (C < 1 || C > 65535) return false;
    int per = (tiles + C - 1) / C;
    if (per > kStreamMaxTiles) {
        if (force_c) return false;
        C = (tiles + kStreamMaxTiles - 1) / kStreamMaxTiles;
        per = (tiles + C - 1) / C;
    }
    auto deepest = [&](int bk_) {   // deepest ring that fits, at most kSplitMaxStages
        int st = kSplitMaxStages;
        while (st > 1 && stream_smem_bytes(M, st, bk_) > kMaxDynSmem) --st;
        return st;
    };
    int bk = force_bk;
    if (!bk) {
        // K in equal chunks of at most 2048 elements; shorter chunks (more of
        // them) until the ring holds two chunks' worth of entries, else one
        int nch = (K + kSplitMaxBK - 1) / kSplitMaxBK;
        int best = 0;
        for (int tries = 0; tries < 6; ++tries, nch *= 2) {
            const int cand = (((K + nch - 1) / nch) + 63) / 64 * 64;
            if (cand < 64) break;
            const int st = deepest(cand);
            if (st >= per + 2) { bk = cand; break; }
            if (!best && st >= per + 1) best = cand;
        }
        if (!bk) bk = best;
    }
    if (bk < 64 || bk > kSplitMaxBK || bk % 64) return false;
    int stages = force_stages ? force_stages : deepest(bk);
    if (stages < per + 1 || stages > kSplitMaxStages) return false;
    const int smem = stream_smem_bytes(M, stages, bk);
    if (smem > kMaxDynSmem) return false;
    p->backend = SKINNY_BACKEND_STREAM;
    p->consumer = SKINNY_CONSUMER_MMA;
    p->vec_elems = 8;
    p->block_n = 16;
    p->split_k = 1;
    p->stages = stages;
    p->stage_k = bk;
    p->k_chunk = K;
    p->grid_x = C;
    p->grid_y = 1;
    p->threads = 160;
    p->smem_bytes = smem;
    return true;
}

// Tensor-core (tcgen05) plan: see tc_make_plan (tmem_gemm.cu).  Rows of X and
// W must be 16-byte aligned (tensor maps).
bool plan_tc(int M, int N, int K, int vec, bool x_ok, int force_bn, int force_s, int force_stages, int force_bk,
             int force_c, int num_sms, skinny_plan_t *p) {
    if (vec != 8 || !x_ok) return false;
    return tc_make_plan(M, N, K, force_bn, force_s, force_stages, force_bk, force_c, num_sms, p);
}

skinny_status_t make_plan(const uint16_t *X, int ldx, const uint16_t *W, int ldw, int M, int N, int K, int num_sms,
                          skinny_plan_t *p) {
    std::memset(p, 0, sizeof(*p));
    if (num_sms < 1) return SKINNY_ERR_INVALID_VALUE;
    const int vec = widest_vec(W, ldw);
    const int fb = g_opt_force_backend.load(), fc = g_opt_force_consumer.load();
    const int fs = g_opt_force_split_k.load(), fbn = g_opt_force_block_n.load();
    const int fst = g_opt_force_stages.load();
    const int fgy = g_opt_force_grid_y.load();
    const bool splitk_ok = vec == 8 && K % 8 == 0;
    const bool mma_ok = splitk_ok && K % 16 == 0;
    const bool x_ok = (reinterpret_cast<uintptr_t>(X) & 15) == 0 && ldx % 8 == 0;
    const bool stream_ok = mma_ok && x_ok && M <= kMaxMSmall;
    const bool tc_ok = vec == 8 && x_ok;

    int backend = fb, consumer = fc, split = fs, bn = fbn, stages = fst, stage_k = g_opt_force_stage_k.load();
    int clusters = fgy;
    int tuned = 0;
    const bool dotmma_ok = splitk_ok && K % 32 == 0;
    // 17..64 tokens: tensor cores only, on the split-K backend, on the
    // tensor-core dot-product for large weights (>= 16 MB, K % 32 == 0), or on
    // the tcgen05 backend (also the only one for K % 16 != 0)
    const bool mid_m = M > kMaxMSmall;
    if (mid_m) {
        if (!mma_ok && !tc_ok) return SKINNY_ERR_UNSUPPORTED;
        if ((fb != SKINNY_BACKEND_AUTO && fb != SKINNY_BACKEND_SPLITK && fb != SKINNY_BACKEND_DOTPROD &&
             fb != SKINNY_BACKEND_TCGEN05) ||
            (fc != SKINNY_CONSUMER_AUTO && fc != SKINNY_CONSUMER_MMA))
            return SKINNY_ERR_UNSUPPORTED;
        consumer = SKINNY_CONSUMER_MMA;
        if (fb == SKINNY_BACKEND_DOTPROD && !dotmma_ok) return SKINNY_ERR_UNSUPPORTED;
        if (fb == SKINNY_BACKEND_SPLITK && !mma_ok) return SKINNY_ERR_UNSUPPORTED;
        backend = fb != SKINNY_BACKEND_AUTO                ? fb
                  : (!mma_ok || (tc_ok && 2.0 * N * K >= 16e6)) ? SKINNY_BACKEND_TCGEN05
                  : (dotmma_ok && 2.0 * N * K >= 16e6)         ? SKINNY_BACKEND_DOTPROD
                                                               : SKINNY_BACKEND_SPLITK;
        const TunedEntry *e = (fb == SKINNY_BACKEND_AUTO) ? lookup_tuned(M, N, K) : nullptr;
        if (e && e->backend == SKINNY_BACKEND_TCGEN05 && tc_ok) {
            backend = SKINNY_BACKEND_TCGEN05;
            if (!bn) bn = e->block_n;
            if (!split) split = e->split_k;
            if (!stages) stages = e->stages;
            if (!stage_k) stage_k = e->stage_k;
            if (!clusters) clusters = e->clusters;
            tuned = 1;
        } else if (e && e->backend == SKINNY_BACKEND_SPLITK && e->consumer == SKINNY_CONSUMER_MMA && mma_ok) {
            backend = SKINNY_BACKEND_SPLITK;
            if (!split) split = e->split_k;
            if (!stages) stages = e->stages;
            if (!stage_k) stage_k = e->stage_k;
            tuned = 1;
        } else if (e && e->backend == SKINNY_BACKEND_DOTPROD && e->consumer == SKINNY_CONSUMER_MMA && dotmma_ok) {
            backend = SKINNY_BACKEND_DOTPROD;
            if (!bn) bn = e->block_n;
            if (!split) split = e->split_k;
            tuned = 1;
        }
    }
    if (backend == SKINNY_BACKEND_AUTO) {
        const TunedEntry *e = lookup_tuned(M, N, K);
        const bool entry_ok =
            e && ((e->backend == SKINNY_BACKEND_DOTPROD && e->consumer != SKINNY_CONSUMER_MMA) ||
                  (e->backend == SKINNY_BACKEND_DOTPROD && e->consumer == SKINNY_CONSUMER_MMA && dotmma_ok) ||
                  (e->backend == SKINNY_BACKEND_SPLITK && splitk_ok &&
                   (e->consumer != SKINNY_CONSUMER_MMA || mma_ok)) ||
                  (e->backend == SKINNY_BACKEND_STREAM && stream_ok) ||
                  (e->backend == SKINNY_BACKEND_TCGEN05 && tc_ok));
        if (entry_ok) {
            backend = e->backend;
            if (consumer == SKINNY_CONSUMER_AUTO) consumer = e->consumer;
            if (!split) split = e->split_k;
            if (!bn) bn = e->block_n;
            if (!stages) stages = e->stages;
            if (!stage_k) stage_k = e->stage_k;
            if (!clusters) clusters = e->clusters;
            tuned = 1;
        } else if (tc_ok && M >= 9 && 2.0 * N * K >= 16e6) {
            // default rule, bandwidth-bound weights (>= 16 MB) and 9..16 tokens:
            // tcgen05 (measured ahead of the other backends there on GB300)
            backend = SKINNY_BACKEND_TCGEN05;
        } else if (dotmma_ok && M >= 4 && 2.0 * N * K >= 16e6) {
            // default rule, bandwidth-bound weights (>= 16 MB): tensor-core dot-product
            backend = SKINNY_BACKEND_DOTPROD;
            if (consumer == SKINNY_CONSUMER_AUTO) consumer = SKINNY_CONSUMER_MMA;
        } else {
            // default rule: dot-product for small M or short K, else split-K
            backend = (M <= 4 || K < 2048 || !splitk_ok) ? SKINNY_BACKEND_DOTPROD : SKINNY_BACKEND_SPLITK;
        }
    }
    bool ok;
    if (backend == SKINNY_BACKEND_DOTPROD && consumer == SKINNY_CONSUMER_MMA) {
        ok = plan_dotmma(M, N, K, vec, bn, split, num_sms, p);
        if (!ok && tuned && fs == 0 && fbn == 0) {
            // a tuned split these sizes cannot take: the one-CTA-per-block plan
            ok = plan_dotmma(M, N, K, vec, 0, 0, num_sms, p);
            tuned = 0;
        }
        if (!ok && fb == SKINNY_BACKEND_AUTO && mid_m) {
            ok = plan_splitk(M, N, K, vec, consumer, fs, fst, fgy, g_opt_force_stage_k.load(), num_sms, p);
            tuned = 0;
        } else if (!ok && fb == SKINNY_BACKEND_AUTO && fc == SKINNY_CONSUMER_AUTO) {
            ok = plan_dotprod(M, N, K, vec, 0, num_sms, p);
            tuned = 0;
        }
    } else if (backend == SKINNY_BACKEND_DOTPROD) {
        if (vec != 8 && bn > 1 && fbn) return SKINNY_ERR_UNSUPPORTED;
        ok = plan_dotprod(M, N, K, vec, vec == 8 ? bn : 1, num_sms, p);
    } else if (backend == SKINNY_BACKEND_SPLITK) {
        if (consumer == SKINNY_CONSUMER_AUTO) consumer = (M > 4 && mma_ok) ? SKINNY_CONSUMER_MMA : SKINNY_CONSUMER_FMA;
        if (bn != 0 && bn != 16) return SKINNY_ERR_UNSUPPORTED;
        ok = plan_splitk(M, N, K, vec, consumer, split, stages, clusters, stage_k, num_sms, p);
        if (!ok && mid_m && tuned) {
            // a tuned entry these pointers / strides cannot use: the default split-K plan
            ok = plan_splitk(M, N, K, vec, consumer, fs, fst, fgy, g_opt_force_stage_k.load(), num_sms, p);
            tuned = 0;
        }
        if (!ok && fb == SKINNY_BACKEND_AUTO && !mid_m) {
            // a tuned split-K entry that these pointers / strides cannot use
            ok = plan_dotprod(M, N, K, vec, 0, num_sms, p);
            tuned = 0;
        }
        if (!ok && fb == SKINNY_BACKEND_AUTO && mid_m && tc_ok) {
            // 17..64 tokens whose X slice does not fit beside the split-K ring
            ok = plan_tc(M, N, K, vec, x_ok, 0, 0, 0, 0, 0, num_sms, p);
            tuned = 0;
        }
    } else if (backend == SKINNY_BACKEND_STREAM) {
        if ((fc != SKINNY_CONSUMER_AUTO && fc != SKINNY_CONSUMER_MMA) || (bn != 0 && bn != 16))
            return SKINNY_ERR_UNSUPPORTED;
        ok = plan_stream(M, N, K, vec, x_ok, clusters, stages, stage_k, num_sms, p);
        if (!ok && fb == SKINNY_BACKEND_AUTO) {
            // a tuned or default streaming plan these pointers / sizes cannot use
            ok = (dotmma_ok && M >= 4 && plan_dotmma(M, N, K, vec, 0, 0, num_sms, p)) ||
                 plan_dotprod(M, N, K, vec, 0, num_sms, p);
            tuned = 0;
        }
    } else if (backend == SKINNY_BACKEND_TCGEN05) {
        if ((fc != SKINNY_CONSUMER_AUTO && fc != SKINNY_CONSUMER_MMA) || (bn != 0 && bn != 128 && bn != 64))
            return SKINNY_ERR_UNSUPPORTED;
        ok = plan_tc(M, N, K, vec, x_ok, bn, split, stages, stage_k, clusters, num_sms, p);
        if (!ok && fb == SKINNY_BACKEND_AUTO) {
            // a tuned tensor-core plan these pointers / strides cannot use: the
            // default rule of the token range
            const bool big = dotmma_ok && 2.0 * N * K >= 16e6;
            ok = mid_m ? ((big && plan_dotmma(M, N, K, vec, 0, 0, num_sms, p)) ||
                          plan_splitk(M, N, K, vec, SKINNY_CONSUMER_MMA, fs, fst, fgy, g_opt_force_stage_k.load(),
                                      num_sms, p))
                       : ((big && M >= 4 && plan_dotmma(M, N, K, vec, 0, 0, num_sms, p)) ||
                          plan_dotprod(M, N, K, vec, 0, num_sms, p));
            tuned = 0;
        }
    } else {
        return SKINNY_ERR_INVALID_VALUE;
    }
    if (!ok) return SKINNY_ERR_UNSUPPORTED;
    p->pdl = pdl_for(2.0 * N * K, p->backend != SKINNY_BACKEND_DOTPROD);
    p->tuned = tuned;
    return SKINNY_OK;
}

void log_plan(int M, int N, int K, int ldw, const skinny_plan_t &p) {
    static std::mutex mu;
    static std::set<std::tuple<int, int, int, int, int>> seen;
    std::lock_guard<std::mutex> g(mu);
    if (!seen.insert({M, N, K, ldw, p.pdl}).second) return;
    std::fprintf(stderr,
                 "[skinny] M=%d N=%d K=%d ldw=%d -> %s consumer=%d vec=%d block_n=%d split_k=%d stages=%d stage_k=%d "
                 "k_chunk=%d grid=%dx%d smem=%d pdl=%d tuned=%d\n",
                 M, N, K, ldw,
                 p.backend == SKINNY_BACKEND_DOTPROD  ? "dotprod"
                 : p.backend == SKINNY_BACKEND_SPLITK ? "splitk"
                 : p.backend == SKINNY_BACKEND_STREAM ? "stream"
                                                      : "tcgen05",
                 p.consumer,
                 p.vec_elems, p.block_n, p.split_k, p.stages, p.stage_k, p.k_chunk, p.grid_x, p.grid_y, p.smem_bytes,
                 p.pdl, p.tuned);
}

}  // namespace
}  // namespace skinny

using namespace skinny;

namespace skinny {
namespace {
// One call: checks, plan, launch.  out_bf16 selects a bf16 Y (2-byte elements).
skinny_status_t run_gemm(const uint16_t *X, int ldx, const uint16_t *W, int ldw, void *Y, int ldy,
                         int M, int N, int K, void *stream, int out_bf16) {
    bool noop = false;
    skinny_status_t st = validate(X, ldx, W, ldw, Y, ldy, M, N, K, &noop, out_bf16 ? 2 : 4);
    if (st != SKINNY_OK || noop) return st;
    int device = 0;
    st = current_device(&device);
    if (st != SKINNY_OK) return st;
    DeviceState &d = g_dev[device];
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) {
        const int64_t total = (int64_t)M * N;
        int blocks = (int)((total + 255) / 256);
        if (blocks > 4 * d.num_sms) blocks = 4 * d.num_sms;
        zero_fill_kernel<<<blocks, 256, 0, s>>>(Y, ldy, M, N, out_bf16);
        return cudaPeekAtLastError() == cudaSuccess ? SKINNY_OK : SKINNY_ERR_LAUNCH;
    }
    skinny_plan_t plan;
    st = make_plan(X, ldx, W, ldw, M, N, K, d.num_sms, &plan);
    if (st != SKINNY_OK) return st;
    if (opt_log()) log_plan(M, N, K, ldw, plan);
    GemmArgs a{X, ldx, W, ldw, Y, ldy, M, N, K, out_bf16};
    LaunchCtx c{s, plan.pdl != 0, late_trigger(2.0 * N * K), d.status_word, (uint64_t)g_opt_wait_us.load() * 1000ull};
    cudaError_t e;
    if (plan.backend == SKINNY_BACKEND_DOTPROD)
        e = plan.consumer == SKINNY_CONSUMER_MMA ? launch_dotmma(a, plan, c) : launch_dotprod(a, plan, c);
    else if (plan.backend == SKINNY_BACKEND_STREAM)
        e = launch_stream(a, plan, c);
    else if (plan.backend == SKINNY_BACKEND_TCGEN05)
        e = launch_tc(a, plan, c);
    else
        e = launch_splitk(a, plan, c);
    return e == cudaSuccess ? SKINNY_OK : SKINNY_ERR_LAUNCH;
}

// fp32 weights, tensor-core dot-product (two tf32 terms per weight): 16-row
// blocks (or the forced block_n), K over a cluster of S CTAs, S the largest
// power of two up to 8 that keeps the grid within two CTAs per SM and gives
// every rank some K (or the forced split_k), the rank's X slice resident.
// Measured on GB300, L2-cold chains, 7168 x 384: 7.1 us at 8 tokens, 8.7 at
// 16 (the CUDA-core kernel 13.0 and 19.4).
bool plan_f32w_mma(int M, int N, int K, int num_sms, int force_bn, int force_s, skinny_plan_t *p) {
    const int bn = force_bn ? force_bn : 16;
    if (!dotmma_f32w_supported(M, bn) || K < 32 || K % 32) return false;
    const int blocks = (N + bn - 1) / bn;
    int S = force_s;
    if (!S) {
        S = 1;
        while (S < kSplitMaxCluster && (int64_t)blocks * S * 2 <= 2 * num_sms && dotmma_f32w_split_ok(K, S * 2))
            S *= 2;
        while (S < kSplitMaxCluster && dotmma_f32w_smem_bytes(M, bn, K, S) > kMaxDynSmem &&
               dotmma_f32w_split_ok(K, S * 2))
            S *= 2;
    }
    if (!dotmma_f32w_split_ok(K, S) || blocks > 65535) return false;
    p->backend = SKINNY_BACKEND_DOTPROD;
    p->consumer = SKINNY_CONSUMER_MMA;
    p->vec_elems = 4;
    p->block_n = bn;
    p->split_k = S;
    p->k_chunk = S > 1 ? dotmma_f32w_k_slice(K, S) : K;
    p->grid_x = S > 1 ? S : blocks;
    p->grid_y = S > 1 ? blocks : 1;
    p->threads = dotmma_f32w_threads(M);
    p->smem_bytes = dotmma_f32w_smem_bytes(M, bn, K, S);
    p->pdl = pdl_for(4.0 * N * K, false);
    return p->smem_bytes <= kMaxDynSmem;
}

// fp32 weights.  From kF32wMmaMinM tokens on weights of kF32wMmaMinWBytes or
// more, when the W rows are 16-byte aligned and K % 32 == 0, the tensor-core
// dot-product; otherwise (or with the FMA
// consumer forced) the CUDA-core dot-product kernel, W loads as wide as the W
// pointer and ldw allow (4 / 2 / 1 fp32), BN rows per CTA as in the bf16 rule.
// Measured on GB300 (L2-cold chains): below 6 tokens, or on weights under
// 4 MB (2880 x 128: 1.5 MB of fp32), the CUDA-core kernel is faster.
constexpr int kF32wMmaMinM = 6;
constexpr double kF32wMmaMinWBytes = 4e6;
bool plan_f32w(const float *W, int ldw, int M, int N, int K, int num_sms, skinny_plan_t *p) {
    std::memset(p, 0, sizeof(*p));
    const uintptr_t w = reinterpret_cast<uintptr_t>(W);
    const int vec = ((w & 15) == 0 && ldw % 4 == 0) ? 4 : ((w & 7) == 0 && ldw % 2 == 0) ? 2 : 1;
    const int fc = g_opt_force_consumer.load();
    const bool mma_fits = vec == 4 && K >= 32 && K % 32 == 0;
    if (fc == SKINNY_CONSUMER_MMA) {
        return mma_fits && plan_f32w_mma(M, N, K, num_sms, g_opt_force_block_n.load(), g_opt_force_split_k.load(), p);
    }
    if (fc == SKINNY_CONSUMER_AUTO && mma_fits && M >= kF32wMmaMinM && 4.0 * N * K >= kF32wMmaMinWBytes &&
        plan_f32w_mma(M, N, K, num_sms, 0, 0, p))
        return true;
    std::memset(p, 0, sizeof(*p));
    int bn = 1;
    if (vec == 4) {
        bn = pow2_floor(N / (2 * num_sms) > 0 ? N / (2 * num_sms) : 1);
        if (bn > 4) bn = 4;
    }
    if (!dotprod_f32w_supported(M, vec, bn)) return false;
    const int k8 = (K + 7) & ~7;
    int kc = (kDotXBudget / (2 * M)) & ~7;
    if (kc >= k8) {
        kc = k8;
    } else {
        kc = (kc / (8 * kDotThreads)) * (8 * kDotThreads);
        if (kc < 8 * kDotThreads) kc = 8 * kDotThreads;
    }
    p->backend = SKINNY_BACKEND_DOTPROD;
    p->consumer = SKINNY_CONSUMER_FMA;
    p->vec_elems = vec;
    p->block_n = bn;
    p->split_k = 1;
    p->k_chunk = kc;
    p->grid_x = (N + bn - 1) / bn;
    p->grid_y = 1;
    p->threads = kDotThreads;
    p->smem_bytes = dotprod_f32w_smem_bytes(M, bn, kc);
    p->pdl = pdl_for(4.0 * N * K, false);
    return p->smem_bytes <= kMaxDynSmem;
}

// Host-only checks of the router epilogue's arguments; *noop when M == 0 or k == 0.
skinny_status_t validate_topk(const float *L, int ldl, int M, int N, int k, const float *Wt, int ldwt,
                              const int32_t *ids, int ldid, bool *noop) {
    *noop = false;
    if (M < 0 || N < 0 || k < 0) return SKINNY_ERR_INVALID_VALUE;
    if (M == 0 || k == 0) { *noop = true; return SKINNY_OK; }
    if (N < 1 || k > N) return SKINNY_ERR_INVALID_VALUE;
    if (N > kTopkMaxN || k > kTopkMaxK || M > 65535) return SKINNY_ERR_UNSUPPORTED;
    if (!L || !Wt || !ids || ldl < N || ldwt < k || ldid < k) return SKINNY_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(L) | reinterpret_cast<uintptr_t>(Wt) | reinterpret_cast<uintptr_t>(ids)) & 3)
        return SKINNY_ERR_MISALIGNED;
    const uintptr_t l0 = reinterpret_cast<uintptr_t>(L), l1 = l0 + (uintptr_t)(((int64_t)(M - 1) * ldl + N) * 4);
    const uintptr_t w0 = reinterpret_cast<uintptr_t>(Wt), w1 = w0 + (uintptr_t)(((int64_t)(M - 1) * ldwt + k) * 4);
    const uintptr_t i0 = reinterpret_cast<uintptr_t>(ids), i1 = i0 + (uintptr_t)(((int64_t)(M - 1) * ldid + k) * 4);
    if (ranges_overlap(w0, w1, l0, l1) || ranges_overlap(i0, i1, l0, l1) || ranges_overlap(w0, w1, i0, i1))
        return SKINNY_ERR_INVALID_VALUE;
    return SKINNY_OK;
}

skinny_status_t run_topk(const float *L, int ldl, int M, int N, int k, int renormalize, float *Wt, int ldwt,
                         int32_t *ids, int ldid, void *stream) {
    int device = 0;
    skinny_status_t st = current_device(&device);
    if (st != SKINNY_OK) return st;
    const cudaError_t e = launch_router_topk(L, ldl, M, N, k, renormalize ? 1 : 0, Wt, ldwt, ids, ldid,
                                             static_cast<cudaStream_t>(stream), opt_pdl() != 0);
    return e == cudaSuccess ? SKINNY_OK : SKINNY_ERR_LAUNCH;
}
}  // namespace
}  // namespace skinny

extern "C" {

skinny_status_t skinny_gemm_bf16_f32w(const uint16_t *X, int ldx, const float *W, int ldw,
                                      float *Y, int ldy, int M, int N, int K, void *stream) {
    bool noop = false;
    skinny_status_t st = validate(X, ldx, W, ldw, Y, ldy, M, N, K, &noop, 4, 4);
    if (st != SKINNY_OK || noop) return st;
    if (M > kMaxMSmall) return SKINNY_ERR_UNSUPPORTED;
    int device = 0;
    st = current_device(&device);
    if (st != SKINNY_OK) return st;
    DeviceState &d = g_dev[device];
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) {
        const int64_t total = (int64_t)M * N;
        int blocks = (int)((total + 255) / 256);
        if (blocks > 4 * d.num_sms) blocks = 4 * d.num_sms;
        zero_fill_kernel<<<blocks, 256, 0, s>>>(Y, ldy, M, N, 0);
        return cudaPeekAtLastError() == cudaSuccess ? SKINNY_OK : SKINNY_ERR_LAUNCH;
    }
    skinny_plan_t plan;
    if (!plan_f32w(W, ldw, M, N, K, d.num_sms, &plan)) return SKINNY_ERR_UNSUPPORTED;
    LaunchCtx c{s, plan.pdl != 0, false, d.status_word, (uint64_t)g_opt_wait_us.load() * 1000ull};
    const cudaError_t e = plan.consumer == SKINNY_CONSUMER_MMA
                              ? launch_dotmma_f32w(X, ldx, W, ldw, Y, ldy, M, N, K, plan, c)
                              : launch_dotprod_f32w(X, ldx, W, ldw, Y, ldy, M, N, K, plan, c);
    return e == cudaSuccess ? SKINNY_OK : SKINNY_ERR_LAUNCH;
}

skinny_status_t skinny_plan_for_f32w(const uint16_t *X, int ldx, const float *W, int ldw, const float *Y, int ldy,
                                     int M, int N, int K, int num_sms, skinny_plan_t *plan) {
    if (!plan || num_sms < 1) return SKINNY_ERR_INVALID_VALUE;
    bool noop = false;
    skinny_status_t st = validate(X, ldx, W, ldw, Y, ldy, M, N, K, &noop, 4, 4);
    if (st != SKINNY_OK) return st;
    if (M > kMaxMSmall) return SKINNY_ERR_UNSUPPORTED;
    if (noop || K == 0) { std::memset(plan, 0, sizeof(*plan)); return SKINNY_OK; }
    return plan_f32w(W, ldw, M, N, K, num_sms, plan) ? SKINNY_OK : SKINNY_ERR_UNSUPPORTED;
}

skinny_status_t skinny_rmsnorm_gemm_bf16(const uint16_t *X, int ldx, const uint16_t *gamma, float eps,
                                         uint16_t *XN, int ldxn, const uint16_t *W, int ldw, float *Y, int ldy,
                                         int M, int N, int K, void *stream) {
    // the GEMM's own checks, with the normalised rows as its X
    bool noop = false;
    skinny_status_t st = validate(XN, ldxn, W, ldw, Y, ldy, M, N, K, &noop, 4);
    if (st != SKINNY_OK || noop) return st;
    if (K == 0) return run_gemm(XN, ldxn, W, ldw, Y, ldy, M, N, K, stream, 0);   // Y = 0, XN untouched
    if (!(eps >= 0.f) || !std::isfinite(eps)) return SKINNY_ERR_INVALID_VALUE;
    if (!X || !gamma || ldx < K) return SKINNY_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(gamma)) & 1) return SKINNY_ERR_MISALIGNED;
    if (M > SKINNY_MAX_M) return SKINNY_ERR_UNSUPPORTED;
    // XN is written: it may overlap none of X, gamma, W or Y
    const uintptr_t n0 = reinterpret_cast<uintptr_t>(XN), n1 = n0 + (uintptr_t)(((int64_t)(M - 1) * ldxn + K) * 2);
    const uintptr_t x0 = reinterpret_cast<uintptr_t>(X), x1 = x0 + (uintptr_t)(((int64_t)(M - 1) * ldx + K) * 2);
    const uintptr_t g0 = reinterpret_cast<uintptr_t>(gamma), g1 = g0 + (uintptr_t)K * 2;
    const uintptr_t w0 = reinterpret_cast<uintptr_t>(W), w1 = w0 + (uintptr_t)(((int64_t)(N - 1) * ldw + K) * 2);
    const uintptr_t y0 = reinterpret_cast<uintptr_t>(Y), y1 = y0 + (uintptr_t)(((int64_t)(M - 1) * ldy + N) * 4);
    if (ranges_overlap(n0, n1, x0, x1) || ranges_overlap(n0, n1, g0, g1) || ranges_overlap(n0, n1, w0, w1) ||
        ranges_overlap(n0, n1, y0, y1) || ranges_overlap(y0, y1, x0, x1) || ranges_overlap(y0, y1, g0, g1))
        return SKINNY_ERR_INVALID_VALUE;
    // the plan must exist before anything is launched
    int device = 0;
    st = current_device(&device);
    if (st != SKINNY_OK) return st;
    DeviceState &d = g_dev[device];
    skinny_plan_t plan;
    st = make_plan(XN, ldxn, W, ldw, M, N, K, d.num_sms, &plan);
    if (st != SKINNY_OK) return st;
    skinny_plan_t fused;
    const bool x_rows_16 = (reinterpret_cast<uintptr_t>(X) & 15) == 0 && ldx % 8 == 0;   // the raw rows by TMA
    if (g_opt_fuse_norm.load() && x_rows_16 && tc_make_norm_plan(M, N, K, plan, &fused)) {
        // one launch: the norm runs inside every CTA of the tcgen05 GEMM
        if (opt_log()) log_plan(M, N, K, ldw, fused);
        GemmArgs a{XN, ldxn, W, ldw, Y, ldy, M, N, K, 0};
        LaunchCtx c{static_cast<cudaStream_t>(stream), plan.pdl != 0, late_trigger(2.0 * N * K), d.status_word,
                    (uint64_t)g_opt_wait_us.load() * 1000ull};
        const TcNormArgs na{X, ldx, gamma, eps, XN, ldxn};
        return launch_tc(a, fused, c, &na) == cudaSuccess ? SKINNY_OK : SKINNY_ERR_LAUNCH;
    }
    const cudaError_t e = launch_rmsnorm(X, ldx, gamma, eps, M, K, XN, ldxn, static_cast<cudaStream_t>(stream),
                                         opt_pdl() != 0);
    if (e != cudaSuccess) return SKINNY_ERR_LAUNCH;
    return run_gemm(XN, ldxn, W, ldw, Y, ldy, M, N, K, stream, 0);
}

skinny_status_t skinny_router_topk(const float *logits, int ldl, int M, int N, int k, int renormalize,
                                   float *weights, int ldw, int32_t *ids, int ldid, void *stream) {
    bool noop = false;
    const skinny_status_t st = validate_topk(logits, ldl, M, N, k, weights, ldw, ids, ldid, &noop);
    if (st != SKINNY_OK || noop) return st;
    return run_topk(logits, ldl, M, N, k, renormalize, weights, ldw, ids, ldid, stream);
}

skinny_status_t skinny_router_bf16_topk(const uint16_t *X, int ldx, const uint16_t *W, int ldw,
                                        float *logits, int ldl, int M, int N, int K, int k, int renormalize,
                                        float *weights, int ldwt, int32_t *ids, int ldid, void *stream) {
    // every argument of both steps is checked before anything is launched
    bool noop_g = false, noop_t = false;
    skinny_status_t st = validate(X, ldx, W, ldw, logits, ldl, M, N, K, &noop_g, 4);
    if (st != SKINNY_OK) return st;
    st = validate_topk(logits, ldl, M, N, k, weights, ldwt, ids, ldid, &noop_t);
    if (st != SKINNY_OK) return st;
    if (!noop_t) {
        const uintptr_t w0 = reinterpret_cast<uintptr_t>(weights), i0 = reinterpret_cast<uintptr_t>(ids);
        const uintptr_t w1 = w0 + (uintptr_t)(((int64_t)(M - 1) * ldwt + k) * 4);
        const uintptr_t i1 = i0 + (uintptr_t)(((int64_t)(M - 1) * ldid + k) * 4);
        if (K > 0) {
            const uintptr_t x0 = reinterpret_cast<uintptr_t>(X), x1 = x0 + (uintptr_t)(((int64_t)(M - 1) * ldx + K) * 2);
            const uintptr_t v0 = reinterpret_cast<uintptr_t>(W), v1 = v0 + (uintptr_t)(((int64_t)(N - 1) * ldw + K) * 2);
            if (ranges_overlap(w0, w1, x0, x1) || ranges_overlap(w0, w1, v0, v1) ||
                ranges_overlap(i0, i1, x0, x1) || ranges_overlap(i0, i1, v0, v1))
                return SKINNY_ERR_INVALID_VALUE;
        }
    }
    st = run_gemm(X, ldx, W, ldw, logits, ldl, M, N, K, stream, 0);
    if (st != SKINNY_OK || noop_t) return st;
    return run_topk(logits, ldl, M, N, k, renormalize, weights, ldwt, ids, ldid, stream);
}

skinny_status_t skinny_gemm_bf16(const uint16_t *X, int ldx, const uint16_t *W, int ldw,
                                 float *Y, int ldy, int M, int N, int K, void *stream) {
    return run_gemm(X, ldx, W, ldw, Y, ldy, M, N, K, stream, 0);
}

skinny_status_t skinny_gemm_bf16_bf16out(const uint16_t *X, int ldx, const uint16_t *W, int ldw,
                                         uint16_t *Y, int ldy, int M, int N, int K, void *stream) {
    return run_gemm(X, ldx, W, ldw, Y, ldy, M, N, K, stream, 1);
}

skinny_status_t skinny_init(int device) { return ensure_device(device); }

skinny_status_t skinny_query_plan(const uint16_t *X, int ldx, const uint16_t *W, int ldw, const float *Y, int ldy,
                                  int M, int N, int K, skinny_plan_t *plan) {
    if (!plan) return SKINNY_ERR_INVALID_VALUE;
    bool noop = false;
    skinny_status_t st = validate(X, ldx, W, ldw, Y, ldy, M, N, K, &noop);
    if (st != SKINNY_OK) return st;
    int device = 0;
    st = current_device(&device);
    if (st != SKINNY_OK) return st;
    if (noop || K == 0) { std::memset(plan, 0, sizeof(*plan)); return SKINNY_OK; }
    return make_plan(X, ldx, W, ldw, M, N, K, g_dev[device].num_sms, plan);
}

skinny_status_t skinny_plan_for(const uint16_t *X, int ldx, const uint16_t *W, int ldw, const float *Y, int ldy,
                                int M, int N, int K, int num_sms, skinny_plan_t *plan) {
    if (!plan) return SKINNY_ERR_INVALID_VALUE;
    bool noop = false;
    skinny_status_t st = validate(X, ldx, W, ldw, Y, ldy, M, N, K, &noop);
    if (st != SKINNY_OK) return st;
    if (noop || K == 0) { std::memset(plan, 0, sizeof(*plan)); return SKINNY_OK; }
    return make_plan(X, ldx, W, ldw, M, N, K, num_sms, plan);
}

skinny_status_t skinny_set_option(int option, int value) {
    switch (option) {
        case SKINNY_OPT_PDL:
            if (value < 0 || value > 2) return SKINNY_ERR_INVALID_VALUE;
            g_opt_pdl.store(value); return SKINNY_OK;
        case SKINNY_OPT_FORCE_BACKEND:
            if (value < 0 || value > 4) return SKINNY_ERR_INVALID_VALUE;
            g_opt_force_backend.store(value); return SKINNY_OK;
        case SKINNY_OPT_FORCE_CONSUMER:
            if (value < 0 || value > 2) return SKINNY_ERR_INVALID_VALUE;
            g_opt_force_consumer.store(value); return SKINNY_OK;
        case SKINNY_OPT_FORCE_SPLIT_K:
            if (value < 0 || value > kSplitMaxCluster) return SKINNY_ERR_INVALID_VALUE;
            g_opt_force_split_k.store(value); return SKINNY_OK;
        case SKINNY_OPT_FORCE_BLOCK_N:
            if (!(value == 0 || value == 1 || value == 2 || value == 4 || value == 8 || value == 16 ||
                  value == 32 || value == 64 || value == 128))
                return SKINNY_ERR_INVALID_VALUE;
            g_opt_force_block_n.store(value); return SKINNY_OK;
        case SKINNY_OPT_FORCE_STAGES:
            if (value < 0 || value > kSplitMaxStages) return SKINNY_ERR_INVALID_VALUE;
            g_opt_force_stages.store(value); return SKINNY_OK;
        case SKINNY_OPT_WAIT_TIMEOUT_US:
            if (value < 0) return SKINNY_ERR_INVALID_VALUE;
            g_opt_wait_us.store(value); return SKINNY_OK;
        case SKINNY_OPT_LOG:
            if (value != 0 && value != 1) return SKINNY_ERR_INVALID_VALUE;
            g_opt_log.store(value); return SKINNY_OK;
        case SKINNY_OPT_FORCE_CLUSTERS:
            if (value < 0 || value > 65535) return SKINNY_ERR_INVALID_VALUE;
            g_opt_force_grid_y.store(value); return SKINNY_OK;
        case SKINNY_OPT_FORCE_STAGE_K:
            if (value < 0 || value > kSplitMaxBK || value % 64) return SKINNY_ERR_INVALID_VALUE;
            g_opt_force_stage_k.store(value); return SKINNY_OK;
        case SKINNY_OPT_FUSE_NORM:
            if (value != 0 && value != 1) return SKINNY_ERR_INVALID_VALUE;
            g_opt_fuse_norm.store(value); return SKINNY_OK;
        case SKINNY_OPT_LATE_TRIGGER:
            if (value != 0 && value != 1) return SKINNY_ERR_INVALID_VALUE;
            g_opt_late_trigger.store(value); return SKINNY_OK;
        default:
            return SKINNY_ERR_INVALID_VALUE;
    }
}

skinny_status_t skinny_get_option(int option, int *value) {
    if (!value) return SKINNY_ERR_INVALID_VALUE;
    switch (option) {
        case SKINNY_OPT_PDL: *value = opt_pdl(); return SKINNY_OK;
        case SKINNY_OPT_FORCE_BACKEND: *value = g_opt_force_backend.load(); return SKINNY_OK;
        case SKINNY_OPT_FORCE_CONSUMER: *value = g_opt_force_consumer.load(); return SKINNY_OK;
        case SKINNY_OPT_FORCE_SPLIT_K: *value = g_opt_force_split_k.load(); return SKINNY_OK;
        case SKINNY_OPT_FORCE_BLOCK_N: *value = g_opt_force_block_n.load(); return SKINNY_OK;
        case SKINNY_OPT_FORCE_STAGES: *value = g_opt_force_stages.load(); return SKINNY_OK;
        case SKINNY_OPT_WAIT_TIMEOUT_US: *value = g_opt_wait_us.load(); return SKINNY_OK;
        case SKINNY_OPT_LOG: *value = opt_log(); return SKINNY_OK;
        case SKINNY_OPT_FORCE_CLUSTERS: *value = g_opt_force_grid_y.load(); return SKINNY_OK;
        case SKINNY_OPT_FORCE_STAGE_K: *value = g_opt_force_stage_k.load(); return SKINNY_OK;
        case SKINNY_OPT_FUSE_NORM: *value = g_opt_fuse_norm.load(); return SKINNY_OK;
        case SKINNY_OPT_LATE_TRIGGER: *value = g_opt_late_trigger.load(); return SKINNY_OK;
        default: return SKINNY_ERR_INVALID_VALUE;
    }
}

skinny_status_t skinny_get_device_status(void *stream, int *code) {
    if (!code) return SKINNY_ERR_INVALID_VALUE;
    int device = 0;
    skinny_status_t st = current_device(&device);
    if (st != SKINNY_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> g(g_status_mu);
    int v = 0;
    status_take_kernel<<<1, 1, 0, s>>>();
    if (cudaPeekAtLastError() != cudaSuccess ||
        cudaMemcpyFromSymbolAsync(&v, g_status_taken, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return SKINNY_ERR_LAUNCH;
    *code = v;
    return SKINNY_OK;
}

const char *skinny_status_string(skinny_status_t s) {
    switch (s) {
        case SKINNY_OK: return "SKINNY_OK";
        case SKINNY_ERR_INVALID_VALUE: return "SKINNY_ERR_INVALID_VALUE";
        case SKINNY_ERR_UNSUPPORTED: return "SKINNY_ERR_UNSUPPORTED";
        case SKINNY_ERR_MISALIGNED: return "SKINNY_ERR_MISALIGNED";
        case SKINNY_ERR_LAUNCH: return "SKINNY_ERR_LAUNCH";
        case SKINNY_ERR_DEVICE_TIMEOUT: return "SKINNY_ERR_DEVICE_TIMEOUT";
        case SKINNY_ERR_NO_DEVICE: return "SKINNY_ERR_NO_DEVICE";
        default: return "SKINNY_ERR_UNKNOWN";
    }
}

int skinny_version(void) { return 100; }

}  // extern "C"
