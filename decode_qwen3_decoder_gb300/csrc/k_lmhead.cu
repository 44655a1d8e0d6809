// Final RMSNorm + tied LM head + greedy argmax for ONE token row ("Dentro de un LLM", Paso 8),
// streaming the [vocab][1024] bf16 embedding through a ring of TMA bulk copies.
//
// At batch 1 the head is a 311 MB read for 1024 MACs per row. The GEMV family reaches ~80% of
// HBM on it: each warp issues its rows' loads, waits for them, reduces, and only then issues
// the next rows. Here a producer warp per CTA (two CTAs per SM) keeps LM_NST stages of 16 rows
// (32 KB) in flight with cp.async.bulk (the TMA engine; the weights depend on nothing computed in the step, so
// the first stages are issued before the dependency wait), and 8 consumer warps reduce each
// stage from shared memory (2 rows per warp) against h held in registers.
//
// The numerics are those of the GEMV's head mode, operation for operation: x + the partials
// in order, the sum of squares per 128-thread layout, h = x * rsqrt(mean + eps) * w in fp32,
// each lane's 32 products in the same order and the same butterfly sum, and the packed
// (value, index) keys, so both kernels give the same logits and ids bit for bit.
//
// It can also end the step (Paso 9's bookkeeping, otherwise a kernel of its own): the CTA
// that finishes last, counted on a word that every launch leaves at zero, writes the greedy
// id and advances the sequence's cached length.
#include "qw_internal.h"

namespace {

constexpr int LM_K = 1024;                   // hidden size served
constexpr int LM_CONS_WARPS = 8;
constexpr int LM_THREADS = (LM_CONS_WARPS + 1) * 32;  // + the producer warp
constexpr int LM_ROWS = 2 * LM_CONS_WARPS;   // rows per stage
constexpr int LM_STAGE = LM_ROWS * LM_K * 2; // 32 KB
constexpr int LM_NST = 3;
constexpr int LM_SMEM = LM_NST * LM_STAGE;
constexpr unsigned long long LM_WAIT_NS = 2000000000ull;

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mb_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mb_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(bar)) : "memory");
}
__device__ __forceinline__ void mb_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)), "r"(bytes) : "memory");
}
// Bounded wait for the phase of parity `par` of a local mbarrier; false after about 2 s.
__device__ __forceinline__ bool mb_wait(uint64_t* bar, uint32_t par) {
    uint32_t done = 0;
    uint64_t t0 = 0;
    for (uint32_t n = 0;; ++n) {
        asm volatile(
            "{\n\t.reg .pred q;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(done)
            : "r"(su32(bar)), "r"(par)
            : "memory");
        if (done) return true;
        if (n == 0) t0 = globaltimer_ns();
        else if ((n & 63) == 0 && globaltimer_ns() - t0 > LM_WAIT_NS) return false;
    }
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     su32(dst)),
                 "l"(src), "r"(bytes), "r"(su32(bar))
                 : "memory");
}
__device__ __forceinline__ void cons_sync() { asm volatile("bar.sync 1, %0;" ::"r"(LM_CONS_WARPS * 32) : "memory"); }
__device__ __forceinline__ float dot8(const uint4 w, const float4 a0, const float4 a1, float acc) {
    acc = fmaf(bf_lo(w.x), a0.x, acc);
    acc = fmaf(bf_hi(w.x), a0.y, acc);
    acc = fmaf(bf_lo(w.y), a0.z, acc);
    acc = fmaf(bf_hi(w.y), a0.w, acc);
    acc = fmaf(bf_lo(w.z), a1.x, acc);
    acc = fmaf(bf_hi(w.z), a1.y, acc);
    acc = fmaf(bf_lo(w.w), a1.z, acc);
    acc = fmaf(bf_hi(w.w), a1.w, acc);
    return acc;
}

struct LmP {
    const float* x;       // residual rows; row rows[0] (or 0) is the token's
    const int* rows;
    const bf16* norm_w;   // final norm [1024]
    float eps;
    const bf16* E;        // [vocab][1024]
    int vocab;
    float* logits;        // optional [vocab]
    unsigned long long* best;  // [1] packed argmax key (atomicMax)
    const float* xadd;    // optional partials [n_add][1024] added to x in order
    int n_add;
    int* status;
    // optional step finalize by the CTA that finishes last (next_id == nullptr: none): the
    // greedy id to next_id[0], best cleared, kv_len[seq] += len_add; done counts finished
    // CTAs (zero between launches, reset by that CTA)
    int32_t* next_id;
    int* kv_len;
    int seq, len_add;
    unsigned int* done;
};

}  // namespace

__global__ void __launch_bounds__(LM_THREADS, 2) k_lmhead1(const __grid_constant__ LmP p) {
    extern __shared__ __align__(128) uint8_t lm_sm[];  // [LM_NST][LM_ROWS][1024] bf16
    __shared__ __align__(8) uint64_t full[LM_NST], empty[LM_NST];
    __shared__ __align__(16) float hs[LM_K];
    __shared__ float red[4];
    __shared__ unsigned long long sbest[LM_CONS_WARPS];
    pdl_launch();
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int nblk = p.vocab / LM_ROWS;
    const int nmine = nblk > (int)blockIdx.x ? (nblk - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    if (t == 0) {
        for (int s = 0; s < LM_NST; ++s) {
            mb_init(&full[s], 1);
            mb_init(&empty[s], LM_CONS_WARPS);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == LM_CONS_WARPS) {
        // ---- producer: stage i holds row block blockIdx.x + i * gridDim.x -----------------
        if (lane == 0) {
            bool ok = true;
            for (int i = 0; i < nmine && ok; ++i) {
                const int s = i % LM_NST;
                if (i >= LM_NST && !mb_wait(&empty[s], (uint32_t)((i / LM_NST - 1) & 1))) {
                    atomicOr(p.status, QW_DEV_TIMEOUT);
                    ok = false;
                    break;
                }
                const size_t blk = (size_t)blockIdx.x + (size_t)i * gridDim.x;
                mb_expect_tx(&full[s], LM_STAGE);
                bulk_g2s(lm_sm + (size_t)s * LM_STAGE, p.E + blk * LM_ROWS * LM_K, LM_STAGE, &full[s]);
            }
            // the copies of the last stages land before the CTA may leave (normally at once)
            for (int i = max(0, nmine - LM_NST); i < nmine; ++i)
                if (!mb_wait(&full[i % LM_NST], (uint32_t)((i / LM_NST) & 1))) break;
        }
        return;
    }

    // ---- consumers: x (+ partials), final RMSNorm into hs (the GEMV's 128-thread layout) ---
    uint2 nwv[2];
    if (t < 128) {
#pragma unroll
        for (int c = 0; c < 2; ++c) nwv[c] = *reinterpret_cast<const uint2*>(p.norm_w + (t + c * 128) * 4);
    }
    pdl_wait();
    if (t < 128) {
        const float* xr = p.x + (size_t)(p.rows ? p.rows[0] : 0) * LM_K;
        float4 v[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) v[c] = *reinterpret_cast<const float4*>(xr + (t + c * 128) * 4);
        for (int g0 = 0; g0 < p.n_add; g0 += 8) {
            float4 a[8][2];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int g = min(g0 + j, p.n_add - 1);
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    a[j][c] = *reinterpret_cast<const float4*>(p.xadd + (size_t)g * LM_K + (t + c * 128) * 4);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (g0 + j < p.n_add) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        v[c].x += a[j][c].x;
                        v[c].y += a[j][c].y;
                        v[c].z += a[j][c].z;
                        v[c].w += a[j][c].w;
                    }
                }
            }
        }
        float part = 0.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            *reinterpret_cast<float4*>(hs + (t + c * 128) * 4) = v[c];
            part += v[c].x * v[c].x + v[c].y * v[c].y + v[c].z * v[c].z + v[c].w * v[c].w;
        }
        part = warp_sum(part);
        if (lane == 0) red[warp] = part;
    }
    cons_sync();
    if (t < 128) {
        const float ss = red[0] + red[1] + red[2] + red[3];
        const float r = rsqrtf(ss / (float)LM_K + p.eps);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            float4* hp = reinterpret_cast<float4*>(hs + (t + c * 128) * 4);
            const float4 v = *hp;
            const uint2 wb = nwv[c];
            *hp = make_float4(v.x * r * bf_lo(wb.x), v.y * r * bf_hi(wb.x), v.z * r * bf_lo(wb.y),
                              v.w * r * bf_hi(wb.y));
        }
    }
    cons_sync();
    // this lane's 32 activations: columns c * 256 + lane * 8 .. + 8, c < 4
    float4 h0[4], h1[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        h0[c] = *reinterpret_cast<const float4*>(hs + c * 256 + lane * 8);
        h1[c] = *reinterpret_cast<const float4*>(hs + c * 256 + lane * 8 + 4);
    }

    // ---- rows: warp w reduces rows 2w, 2w + 1 of every stage ---------------------------
    unsigned long long best = 0ull;
    for (int i = 0; i < nmine; ++i) {
        const int s = i % LM_NST;
        if (!mb_wait(&full[s], (uint32_t)((i / LM_NST) & 1))) {
            if (lane == 0) atomicOr(p.status, QW_DEV_TIMEOUT);
            break;
        }
        const int row0 = (blockIdx.x + i * gridDim.x) * LM_ROWS;
        const bf16* st = reinterpret_cast<const bf16*>(lm_sm + (size_t)s * LM_STAGE);
        uint4 w[2][4];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                w[rr][c] = *reinterpret_cast<const uint4*>(st + (2 * warp + rr) * LM_K + c * 256 + lane * 8);
        __syncwarp();
        if (lane == 0) mb_arrive(&empty[s]);  // the stage is in registers: it may be refilled
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) acc = dot8(w[rr][c], h0[c], h1[c], acc);
            acc = warp_sum(acc);
            const int row = row0 + 2 * warp + rr;
            if (lane == 0) {
                if (p.logits) p.logits[row] = acc;
                best = u64_max(best, argmax_key(acc, row));
            }
        }
    }
    if (lane == 0) sbest[warp] = best;
    cons_sync();
    if (t == 0) {
        unsigned long long b = 0ull;
        for (int w2 = 0; w2 < LM_CONS_WARPS; ++w2) b = u64_max(b, sbest[w2]);
        atomicMax(p.best, b);
        if (p.next_id) {
            // every CTA's maximum is in before its count; the last to count sees them all
            __threadfence();
            if (atomicAdd(p.done, 1u) == gridDim.x - 1) {
                __threadfence();
                const unsigned long long key = atomicExch(p.best, 0ull);
                p.next_id[0] = (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
                p.kv_len[p.seq] += p.len_add;
                atomicExch(p.done, 0u);
            }
        }
    }
}

bool lmhead1_ok(int K, int vocab) { return K == LM_K && vocab % LM_ROWS == 0; }

cudaError_t launch_lmhead1(const LaunchCtx& c, const float* x, const int* rows, const bf16* norm_w, float eps,
                           const bf16* E, int vocab, int K, float* logits, unsigned long long* best,
                           const float* xadd, int n_add, int* status, int num_sms, int32_t* next_id, int* kv_len,
                           int seq, int len_add, unsigned int* done) {
    if (!lmhead1_ok(K, vocab)) return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_lmhead1, cudaFuncAttributeMaxDynamicSharedMemorySize, LM_SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    LmP p = {};
    p.x = x;
    p.rows = rows;
    p.norm_w = norm_w;
    p.eps = eps;
    p.E = E;
    p.vocab = vocab;
    p.logits = logits;
    p.best = best;
    p.xadd = xadd;
    p.n_add = xadd ? n_add : 0;
    p.status = status;
    p.next_id = next_id;
    p.kv_len = kv_len;
    p.seq = seq;
    p.len_add = len_add;
    p.done = done;
    const int grid = std::min(2 * (num_sms > 0 ? num_sms : 148), vocab / LM_ROWS);
    return launch_k(c, k_lmhead1, dim3(grid), dim3(LM_THREADS), (size_t)LM_SMEM, p);
}
