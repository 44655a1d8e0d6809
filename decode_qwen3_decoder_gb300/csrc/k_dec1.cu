// Batch-1 decode layer as two cluster kernels ("Dentro de un LLM: Inferencia en Python puro
// para Qwen3-0.6B en MLX", Pasos 5-7): one new token of one sequence over a short cache.
//
// At batch 1 a layer reads 31.5 MB of weights but is a chain of dependent matrix-vector
// products; as four launches (q|k|v, attention + o_proj, gate/up, down_proj) every link
// pays a kernel hand-off plus an L2 round trip for its input. Here the chain is cut at the
// two places where a result must be gathered from the whole GPU, and every other exchange
// stays inside a thread-block cluster (distributed shared memory):
//
//  k_dec1_attn  one cluster per KV head g (grid n_kv x 16). Each CTA rebuilds x (the layer
//               input: x + the previous layer's down_proj partials, in a fixed order), its
//               RMSNorm, and 32 of the 512 q|k|v rows of head g (q of heads 2g and 2g+1, k, v
//               of g). The 32 results go to every CTA of the cluster; once all 512 have
//               landed each CTA holds q, k, v of head g and runs QK-norm,
//               RoPE and the attention over the cached pages plus the new key (rank 0 also
//               appends K/V to the cache), then o_proj rows [64 r, 64 r + 64) over head g's 256
//               inputs into opart[g]. Cluster 0 writes x.
//  k_dec1_mlp   16 clusters x 8 CTAs; CTA (c, r) owns 24 consecutive intermediate units:
//               x + sum_g opart[g] (fixed order), RMSNorm, its 24 gate and 24 up rows, SwiGLU
//               (fp16-rounded as the activation is stored), then the split-K product of
//               down_proj over those 24 inputs for all 1024 outputs. The 8 partial vectors of a
//               cluster are summed through distributed shared memory (CTA r adds rows
//               [128 r, 128 r + 128) over ranks 0..7 in order) and added into slot c / 2 of
//               dpart. Cluster 0 writes x + sum opart.
//
// The next kernel adds the 8 down_proj slots to x itself, so a layer is two launches. A slot
// takes exactly two atomic adds onto zero (the attention kernel of the same layer clears the
// set, and two sets alternate by layer so that it never clears one still being read); with
// two addends the sum is the same in either order, so the step stays deterministic while
// the reader loads 8 vectors instead of 16.
// The MLP clusters are 8 CTAs so that both kernels' clusters fit on the GPU together (a
// 16-CTA cluster needs 16 free CTA slots in one GPC), which lets each kernel's CTAs start and
// fetch their weights while the other kernel runs.
//
// Exchanges inside a cluster are pushes: st.async into the receiving CTA's shared memory,
// completing bytes on its mbarrier (initialised before the dependency wait and published by
// a relaxed cluster barrier), so no fence sits on the critical path; every wait on an
// mbarrier is bounded and reports QW_DEV_TIMEOUT.
// Nothing read before griddepcontrol.wait is written by an earlier kernel of the step: the
// weights (q|k|v and gate/up rows in registers; o_proj, extra gate/up and down_proj rows and
// the cached K/V pages bulk-copied into shared memory by one thread, cp.async.bulk on an
// mbarrier), the norm weights, the cached length and page table. Every reduction has a fixed
// order (or, for the paired slots, two commuting addends), so a step is deterministic.
#include "qw_internal.h"

namespace {

constexpr int D1_D = 1024;               // hidden size served
constexpr int D1_CL = 16;                // CTAs per cluster
constexpr int D1_THREADS = 256;
constexpr int D1_WARPS = D1_THREADS / 32;
constexpr int D1_MAXPG = 8;              // cached 16-key pages held in shared memory (128 keys)
constexpr int D1_PAGE = 16 * 128 * 2;    // bytes of K (or V) of one page of one KV head
constexpr int D1_CLM = 8;                // CTAs per cluster of the MLP kernel
constexpr int D1_NB = 16;                // clusters of the MLP kernel
constexpr int D1_NP = D1_NB / 2;         // down_proj partials: clusters 2k, 2k + 1 add into slot k
constexpr int D1_ROWS_O = D1_D / D1_CL;  // o_proj rows per CTA (64)
constexpr int D1_ROWS_M = D1_D / D1_CLM; // down_proj rows each MLP CTA sums (128)
constexpr unsigned long long D1_WAIT_NS = 2000000000ull;
constexpr int D1_TRACE_CTAS = 128;       // trace records per launch (both grids have <= 128 CTAs)

// attention kernel, dynamic shared memory: o_proj slice [64][256] bf16 | cached pages
// [D1_MAXPG][K 4 KB | V 4 KB] | h [1024] fp32 | gathered q|k|v of the head [512] fp32
constexpr int A_WO = 0;
constexpr int A_PG = A_WO + D1_ROWS_O * 256 * 2;
constexpr int A_HS = A_PG + D1_MAXPG * 2 * D1_PAGE;
constexpr int A_QKV = A_HS + D1_D * 4;
constexpr int A_SMEM = A_QKV + 512 * 4;

// MLP kernel, dynamic shared memory: gate/up rows not held in registers [2 NS][1024] bf16 |
// transposed down_proj rows [NA][1024] bf16 | h [1024] fp32 | received partial slices
// [8 ranks][128] fp32
template <int NA>
constexpr int mlp_smem() {
    return 2 * (NA - 16) * D1_D * 2 + NA * D1_D * 2 + 2 * D1_D * 4;
}

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
// Bulk copy (TMA engine, not the SM's load/store pipeline) of `bytes` (a multiple of 16, both
// addresses 16-byte aligned) into shared memory, completing on a local mbarrier.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     su32(dst)),
                 "l"(src), "r"(bytes), "r"(su32(bar))
                 : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
// Cluster barrier in two halves (all threads of all CTAs of the cluster): the arrive is
// relaxed, the wait acquires; used once per kernel to publish the mbarrier initialisation.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
// mbarrier expecting `bytes` of remote stores in its first phase (one local arrival)
__device__ __forceinline__ void mbar_init_tx(uint64_t* bar, uint32_t bytes) {
    const uint32_t b = su32(bar);
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b) : "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(bytes) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// 16 bytes into CTA `rank`'s shared memory at the same offset as local address `laddr`,
// counted on that CTA's mbarrier at the same offset as local `lbar`
__device__ __forceinline__ void st_async_f4(uint32_t laddr, uint32_t lbar, uint32_t rank, float4 v) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     map_rank(laddr, rank)),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(map_rank(lbar, rank))
                 : "memory");
}
// Bounded wait for the first phase of a local mbarrier; false after about 2 s.
__device__ __forceinline__ bool mbar_wait0(uint64_t* bar) {
    const uint32_t b = su32(bar);
    uint32_t done = 0;
    uint64_t t0 = 0;
    for (uint32_t n = 0;; ++n) {
        asm volatile(
            "{\n\t.reg .pred q;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 q, [%1], 0;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(done)
            : "r"(b)
            : "memory");
        if (done) return true;
        if (n == 0) t0 = globaltimer_ns();
        else if ((n & 63) == 0 && globaltimer_ns() - t0 > D1_WAIT_NS) return false;
    }
}
// weight fetch issued in program order, so that it stays ahead of griddepcontrol.wait
__device__ __forceinline__ uint4 ldg_w(const void* ptr) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(ptr));
    return r;
}
// 8 bf16 weights (widened exactly) against 8 fp32 activations
__device__ __forceinline__ float dot8w(const uint4 w, const float4 a0, const float4 a1, float acc) {
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
// q . k over this lane's 8 dimensions (fp16 key)
__device__ __forceinline__ float dot8h(const float* q, const uint4 k) {
    const uint32_t w[4] = {k.x, k.y, k.z, k.w};
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        acc = fmaf(q[2 * j], h_lo(w[j]), acc);
        acc = fmaf(q[2 * j + 1], h_hi(w[j]), acc);
    }
    return acc;
}
__device__ __forceinline__ float half_sum(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }
// inspection: thread 0 of the CTA records %globaltimer in slot k of its 8 (when tr != NULL)
__device__ __forceinline__ void trace_at(unsigned long long* tr, int k) {
    if (tr && threadIdx.x == 0) tr[k] = globaltimer_ns();
}

// x = xin + sum_{c < n_add} part[c] (added in order of c), then h = x * rsqrt(mean(x^2) + eps) * w
// into hs; thread t owns x[4t .. 4t + 4). Returns this thread's x.
// NMAX: the most partials (n_add <= NMAX), all loaded in one round trip.
template <int NMAX>
__device__ __forceinline__ float4 stage_norm(const float* xin, const float* part, int n_add, uint2 wv, float eps,
                                             float* hs, float* red) {
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    float4 v = *reinterpret_cast<const float4*>(xin + 4 * t);
    if (n_add > 0) {
        float4 a[NMAX];
#pragma unroll
        for (int c = 0; c < NMAX; ++c)
            a[c] = *reinterpret_cast<const float4*>(part + (size_t)min(c, n_add - 1) * D1_D + 4 * t);
#pragma unroll
        for (int c = 0; c < NMAX; ++c) {
            if (c < n_add) {
                v.x += a[c].x;
                v.y += a[c].y;
                v.z += a[c].z;
                v.w += a[c].w;
            }
        }
    }
    const float ss = warp_sum(v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < D1_WARPS; ++w) tot += red[w];
    const float r = rsqrtf(tot / (float)D1_D + eps);
    *reinterpret_cast<float4*>(hs + 4 * t) =
        make_float4(v.x * r * bf_lo(wv.x), v.y * r * bf_hi(wv.x), v.z * r * bf_lo(wv.y), v.w * r * bf_hi(wv.y));
    return v;
}

}  // namespace

__global__ void __launch_bounds__(D1_THREADS, 2) k_dec1_attn(const __grid_constant__ Dec1Attn p) {
    extern __shared__ __align__(128) uint8_t d1_sm[];
    __shared__ float red[D1_WARPS];
    __shared__ float so[D1_WARPS][128];  // per-warp partial output of its head
    __shared__ float smm[D1_WARPS], sll[D1_WARPS];
    __shared__ __align__(8) uint64_t bar_g;  // the head's 512 gathered q|k|v values have landed
    __shared__ __align__(8) uint64_t bar_w;  // the o_proj slice and the cached pages have landed
    __shared__ int s_np, s_bad;
    pdl_launch();
    unsigned long long* tr = p.trace ? p.trace + ((size_t)2 * p.layer * D1_TRACE_CTAS + blockIdx.x) * 8 : nullptr;
    trace_at(tr, 0);
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int rank = (int)cluster_rank(), g = (int)cluster_id();
    bf16* wo_s = reinterpret_cast<bf16*>(d1_sm + A_WO);
    uint8_t* pg_s = d1_sm + A_PG;
    float* hs = reinterpret_cast<float*>(d1_sm + A_HS);
    float* qkv_s = reinterpret_cast<float*>(d1_sm + A_QKV);
    // reuses (so that two CTAs fit per SM): h is dead once the q|k|v products are reduced,
    // the gathered q|k|v once QK-norm has read it
    float(*sq)[128] = reinterpret_cast<float(*)[128]>(hs);         // rotated q of heads 2g, 2g+1
    float(*skv)[128] = reinterpret_cast<float(*)[128]>(hs + 256);  // the new k (rotated) and v, fp16 values
    float* ob = qkv_s;  // [256] attention output of heads 2g, 2g+1 (fp16 values)
    const f16* Kl = p.kv.k + (size_t)p.layer * p.kv.layer_stride;
    const f16* Vl = p.kv.v + (size_t)p.layer * p.kv.layer_stride;
    const int* pt = p.kv.page_table + (size_t)p.seq * p.kv.max_pages_per_seq;

    // ---- before the wait --------------------------------------------------------------
    // one thread issues the bulk copies: the o_proj rows [64 rank, +64) over inputs
    // [256 g, +256) (64 rows of 512 bytes) and the cached K/V pages of head g (the length and
    // page table were set before the step began)
    if (t == 0) {
        const int cached = p.kv.len[p.seq];
        const int np = min((cached + 15) >> 4, D1_MAXPG);
        mbar_init_tx(&bar_w, (uint32_t)(D1_ROWS_O * 512 + np * 2 * D1_PAGE));
        for (int r = 0; r < D1_ROWS_O; ++r)
            bulk_g2s(wo_s + r * 256, p.Wo + (size_t)(D1_ROWS_O * rank + r) * p.QD + 256 * g, 512, &bar_w);
        int bad = 0, pages[D1_MAXPG];
#pragma unroll
        for (int pi = 0; pi < D1_MAXPG; ++pi) pages[pi] = pi < np ? pt[pi] : 0;  // loads in flight together
#pragma unroll
        for (int pi = 0; pi < D1_MAXPG; ++pi) {
            if (pi >= np) break;
            int page = pages[pi];
            if (page < 0 || page >= p.kv.n_pages) {
                bad = 1;  // no copy from outside the pool; the attention is skipped and reported
                page = 0;
            }
            const size_t off = ((size_t)page * p.n_kv + g) * 16 * 128;
            bulk_g2s(pg_s + pi * 2 * D1_PAGE, Kl + off, D1_PAGE, &bar_w);
            bulk_g2s(pg_s + pi * 2 * D1_PAGE + D1_PAGE, Vl + off, D1_PAGE, &bar_w);
        }
        s_np = np;
        s_bad = bad;
    }
    // q|k|v rows of head g held by this CTA: local rows [32 rank, +32) of the head's 512
    // (q of heads 2g, 2g+1 = rows 0..255, then k = 256..383, then v = 384..511)
    uint4 wq[4][4];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        const int lr = 32 * rank + 4 * warp + rr;
        const int row = lr < 256 ? 256 * g + lr
                                 : (lr < 384 ? p.QD + 128 * g + (lr - 256) : p.QD + p.KD + 128 * g + (lr - 384));
#pragma unroll
        for (int c = 0; c < 4; ++c) wq[rr][c] = ldg_w(p.Wqkv + (size_t)row * D1_D + c * 256 + lane * 8);
    }
    const uint2 wn = *reinterpret_cast<const uint2*>(p.w_in + 4 * t);
    const uint2 wqk = *reinterpret_cast<const uint2*>((warp < 2 ? p.q_norm : p.k_norm) + lane * 4);
    if (t == 0) mbar_init_tx(&bar_g, 512 * 4);
    cluster_arrive_relaxed();
    pdl_wait();
    trace_at(tr, 1);
    // the partial set this layer's MLP kernel adds into starts at zero; its last reader (the
    // attention kernel of the layer before, or the LM head of the step before) has completed
    {
        const int i = blockIdx.x * D1_THREADS + t;
        if (i < D1_NP * D1_D / 4) reinterpret_cast<float4*>(p.dclear)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // the token's position and its RoPE row (in flight while x is staged)
    const int pos = p.pos[0];
    const int i0 = (lane & 15) * 4;
    const float4 cs = *reinterpret_cast<const float4*>(p.rope_cos + (size_t)pos * 64 + i0);
    const float4 sn = *reinterpret_cast<const float4*>(p.rope_sin + (size_t)pos * 64 + i0);

    // ---- x, RMSNorm, q|k|v --------------------------------------------------------------
    const float4 xv = stage_norm<D1_NP>(p.xin, p.dpart, p.n_add, wn, p.eps, hs, red);
    if (g == 0 && (t >> 4) == rank) *reinterpret_cast<float4*>(p.xout + 4 * t) = xv;
    cluster_wait();  // every CTA's mbarrier is initialised
    __syncthreads();
    trace_at(tr, 2);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float4 a0 = *reinterpret_cast<const float4*>(hs + c * 256 + lane * 8);
        const float4 a1 = *reinterpret_cast<const float4*>(hs + c * 256 + lane * 8 + 4);
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) acc[rr] = dot8w(wq[rr][c], a0, a1, acc[rr]);
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) acc[rr] = warp_sum(acc[rr]);
    // all-gather of the head's 512 values: lane L pushes this warp's four rows into CTA L
    if (lane < D1_CL)
        st_async_f4(su32(qkv_s + 32 * rank + 4 * warp), su32(&bar_g), (uint32_t)lane,
                    make_float4(acc[0], acc[1], acc[2], acc[3]));
    if (!mbar_wait0(&bar_g) && t == 0) atomicOr(p.status, QW_DEV_TIMEOUT);
    trace_at(tr, 3);

    // ---- QK-norm + RoPE of the query heads (warps 0, 1) and the new key (warp 2); v (warp 3)
    if (warp < 4) {
        const float4 xq = *reinterpret_cast<const float4*>(qkv_s + warp * 128 + lane * 4);
        float y[4] = {xq.x, xq.y, xq.z, xq.w};
        if (warp < 3) {
            const float ss = warp_sum(y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3]);
            const float r = rsqrtf(ss * (1.0f / 128.0f) + p.eps);
            const uint2 wb = wqk;
            y[0] *= r * bf_lo(wb.x);
            y[1] *= r * bf_hi(wb.x);
            y[2] *= r * bf_lo(wb.y);
            y[3] *= r * bf_hi(wb.y);
            // rotate-half RoPE: dimension i pairs with i + 64 (lanes L and L ^ 16)
            const float cv[4] = {cs.x, cs.y, cs.z, cs.w}, sv[4] = {sn.x, sn.y, sn.z, sn.w};
            float o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float pj = __shfl_xor_sync(0xffffffffu, y[j], 16);
                o[j] = (lane < 16) ? (y[j] * cv[j] - pj * sv[j]) : (pj * sv[j] + y[j] * cv[j]);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) y[j] = o[j];
        }
        if (warp < 2) {
#pragma unroll
            for (int j = 0; j < 4; ++j) sq[warp][lane * 4 + j] = y[j];
        } else {
            const uint32_t w0 = pack_h2(y[0], y[1]), w1 = pack_h2(y[2], y[3]);
            skv[warp - 2][lane * 4 + 0] = h_lo(w0);
            skv[warp - 2][lane * 4 + 1] = h_hi(w0);
            skv[warp - 2][lane * 4 + 2] = h_lo(w1);
            skv[warp - 2][lane * 4 + 3] = h_hi(w1);
            if (rank == 0) {  // one CTA per KV head appends
                const int pi = pos >> 4;
                const int page = (pi < p.kv.max_pages_per_seq) ? pt[pi] : -1;
                if (page < 0 || page >= p.kv.n_pages) {
                    if (lane == 0) atomicOr(p.status, QW_DEV_BAD_POS);
                } else {
                    f16* pool = (warp == 2 ? p.kv.k : p.kv.v) + (size_t)p.layer * p.kv.layer_stride;
                    if (f16_out_of_range(y[0]) || f16_out_of_range(y[1]) || f16_out_of_range(y[2]) ||
                        f16_out_of_range(y[3]))
                        atomicOr(p.status, QW_DEV_RANGE);
                    *reinterpret_cast<uint2*>(pool + (((size_t)page * p.n_kv + g) * 16 + (pos & 15)) * 128 + lane * 4) =
                        make_uint2(w0, w1);
                    if (p.dbg_pos && warp == 2 && g == 0 && lane == 0) {
                        p.dbg_pos[0] = pos;
                        p.dbg_slot[0] = page * 16 + (pos & 15);
                    }
                }
            }
        }
    }
    if (!mbar_wait0(&bar_w) && t == 0) atomicOr(p.status, QW_DEV_TIMEOUT);
    __syncthreads();
    const int np = s_np, bad = s_bad;
    trace_at(tr, 4);
    if (bad && t == 0 && rank == 0) atomicOr(p.status, QW_DEV_BAD_POS);

    // ---- online softmax over the cached keys [0, pos): warp w serves head 2g + (w & 1) on
    //      pages w/2, w/2 + 4 (the page of the new position only below it); the new key goes
    //      to the warp of the head with the fewest pages
    const int hh = warp & 1;
    const int half = lane >> 4, dl = (lane & 15) * 8;
    float q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = sq[hh][dl + i] * p.scale_log2;
    float m = -INFINITY, l = 0.f, o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = 0.f;
    for (int pg = warp >> 1; pg < np && !bad; pg += D1_WARPS / 2) {
        const int nvalid = min(16, pos - pg * 16);
        const uint8_t* kp = pg_s + (size_t)pg * 2 * D1_PAGE;
        uint4 kr[8], vr[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            kr[i] = *reinterpret_cast<const uint4*>(kp + ((2 * i + half) * 128 + dl) * 2);
            vr[i] = *reinterpret_cast<const uint4*>(kp + D1_PAGE + ((2 * i + half) * 128 + dl) * 2);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (2 * i + half >= nvalid) vr[i] = make_uint4(0u, 0u, 0u, 0u);
        float sc[8], pm = -INFINITY;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float d = half_sum(dot8h(q, kr[i]));
            sc[i] = (2 * i + half) < nvalid ? d : -INFINITY;
            pm = fmaxf(pm, sc[i]);
        }
        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
        const float n = fmaxf(m, pm);
        if (n == -INFINITY) continue;
        const float a = exp2f(m - n);
        m = n;
        l *= a;
#pragma unroll
        for (int d = 0; d < 8; ++d) o[d] *= a;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float e = exp2f(sc[i] - m);
            l += e;
            const uint32_t vw[4] = {vr[i].x, vr[i].y, vr[i].z, vr[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                o[2 * j] = fmaf(e, h_lo(vw[j]), o[2 * j]);
                o[2 * j + 1] = fmaf(e, h_hi(vw[j]), o[2 * j + 1]);
            }
        }
    }
    trace_at(tr, 5);
    if (warp == hh + 2 * (np & 3)) {
        // the new key: both half-warps move the max, half 0 adds its weight
        float d = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) d = fmaf(q[i], skv[0][dl + i], d);
        d = half_sum(d);
        const float n = fmaxf(m, d);
        const float a = exp2f(m - n);
        m = n;
        l *= a;
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] *= a;
        if (half == 0) {
            const float e = exp2f(d - m);
            l += e;
#pragma unroll
            for (int j = 0; j < 8; ++j) o[j] = fmaf(e, skv[1][dl + j], o[j]);
        }
    }
    trace_at(tr, 6);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
#pragma unroll
    for (int d = 0; d < 8; ++d) o[d] += __shfl_xor_sync(0xffffffffu, o[d], 16);
    if (lane < 16) {
#pragma unroll
        for (int d = 0; d < 8; ++d) so[warp][dl + d] = o[d];
    }
    if (lane == 0) {
        smm[warp] = m;
        sll[warp] = l;
    }
    __syncthreads();
    {
        // thread -> (head h, dimension d) over the four warps of that head, in order; warps
        // without keys add nothing
        const int h = t >> 7, d = t & 127;
        float M = -INFINITY;
#pragma unroll
        for (int j = 0; j < 4; ++j) M = fmaxf(M, smm[h + 2 * j]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int w = h + 2 * j;
            const float f = smm[w] == -INFINITY ? 0.f : exp2f(smm[w] - M);
            L += sll[w] * f;
            O += so[w][d] * f;
        }
        const __half oh = __float2half_rn(O / L);  // the attention output as the unfused path stores it
        ob[h * 128 + d] = __half2float(oh);
        if (p.dbg_attn && rank == 0) p.dbg_attn[(size_t)(2 * g + h) * 128 + d] = oh;
    }
    __syncthreads();
    // ---- o_proj rows [64 rank, +64) over head g's 256 inputs -------------------------
    const float4 a0 = *reinterpret_cast<const float4*>(&ob[lane * 8]);
    const float4 a1 = *reinterpret_cast<const float4*>(&ob[lane * 8 + 4]);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int lrow = 8 * warp + r;
        const uint4 w = *reinterpret_cast<const uint4*>(wo_s + lrow * 256 + lane * 8);
        const float s = warp_sum(dot8w(w, a0, a1, 0.f));
        if (lane == 0) p.opart[(size_t)g * D1_D + D1_ROWS_O * rank + lrow] = s;
    }
    trace_at(tr, 7);
}

// NA intermediate units per CTA (128 CTAs x NA = inter): 16 from gate/up rows held in
// registers (two per warp), NS = NA - 16 from rows in shared memory (NS / 8 per warp).
template <int NA>
__global__ void __launch_bounds__(D1_THREADS, 2) k_dec1_mlp(const __grid_constant__ Dec1Mlp p) {
    constexpr int NS = NA - 16;
    constexpr int NSW = NS / 8;
    static_assert(NS >= 0 && NS % 8 == 0, "units per CTA: 16, 24 or 32");
    extern __shared__ __align__(128) uint8_t d1_sm[];
    bf16* gu_s = reinterpret_cast<bf16*>(d1_sm);                      // [2 NS][1024]
    bf16* wd_s = reinterpret_cast<bf16*>(d1_sm + 2 * NS * D1_D * 2);  // [NA][1024]
    float* hs = reinterpret_cast<float*>(d1_sm + 2 * NS * D1_D * 2 + NA * D1_D * 2);
    float* rbuf = hs + D1_D;  // [source rank][128]: the other CTAs' partials of this CTA's rows
    __shared__ float red[D1_WARPS];
    __shared__ float sact[NA];
    __shared__ __align__(8) uint64_t bar_r;  // all 8 partial slices have landed
    __shared__ __align__(8) uint64_t bar_w;  // the shared-memory weight rows have landed
    pdl_launch();
    unsigned long long* tr = p.trace ? p.trace + ((size_t)(2 * p.layer + 1) * D1_TRACE_CTAS + blockIdx.x) * 8 : nullptr;
    trace_at(tr, 0);
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int rank = (int)cluster_rank(), c = (int)cluster_id();
    const int a0 = (c * D1_CLM + rank) * NA;  // first intermediate unit of this CTA

    // ---- before the wait: weights ----------------------------------------------------
    if (t == 0) {  // one thread issues the bulk copies of the rows kept in shared memory
        mbar_init_tx(&bar_w, (uint32_t)((2 * NS + NA) * D1_D * 2));
        for (int r = 0; r < 2 * NS; ++r)
            bulk_g2s(gu_s + r * D1_D, (r < NS ? p.Wg : p.Wu) + (size_t)(a0 + 16 + (NS > 0 ? r % NS : 0)) * D1_D,
                     D1_D * 2, &bar_w);
        for (int r = 0; r < NA; ++r) bulk_g2s(wd_s + r * D1_D, p.WdT + (size_t)(a0 + r) * D1_D, D1_D * 2, &bar_w);
    }
    // registers: gate rows a0 + 2w, a0 + 2w + 1 and the same up rows
    uint4 wr[4][4];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        const bf16* W = rr < 2 ? p.Wg : p.Wu;
        const int row = a0 + 2 * warp + (rr & 1);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) wr[rr][ch] = ldg_w(W + (size_t)row * D1_D + ch * 256 + lane * 8);
    }
    const uint2 wn = *reinterpret_cast<const uint2*>(p.w_post + 4 * t);
    if (t == 0) mbar_init_tx(&bar_r, D1_CLM * D1_ROWS_M * 4);
    cluster_arrive_relaxed();
    pdl_wait();
    trace_at(tr, 1);

    // ---- x + o_proj partials, RMSNorm, gate/up, SwiGLU -------------------------------
    const float4 xv = stage_norm<8>(p.xin, p.opart, p.n_add, wn, p.eps, hs, red);
    if (c == 0 && (t >> 5) == rank) *reinterpret_cast<float4*>(p.xout + 4 * t) = xv;
    trace_at(tr, 2);
    if (!mbar_wait0(&bar_w) && t == 0) atomicOr(p.status, QW_DEV_TIMEOUT);
    __syncthreads();
    trace_at(tr, 3);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float accs[2 * NSW > 0 ? 2 * NSW : 1];
#pragma unroll
    for (int k = 0; k < 2 * NSW; ++k) accs[k] = 0.f;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
        const float4 h0 = *reinterpret_cast<const float4*>(hs + ch * 256 + lane * 8);
        const float4 h1 = *reinterpret_cast<const float4*>(hs + ch * 256 + lane * 8 + 4);
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) acc[rr] = dot8w(wr[rr][ch], h0, h1, acc[rr]);
#pragma unroll
        for (int k = 0; k < NSW; ++k) {
            const int u = k * 8 + warp;  // shared-memory unit of this warp
            const uint4 wgt = *reinterpret_cast<const uint4*>(gu_s + u * D1_D + ch * 256 + lane * 8);
            const uint4 wup = *reinterpret_cast<const uint4*>(gu_s + (NS + u) * D1_D + ch * 256 + lane * 8);
            accs[2 * k] = dot8w(wgt, h0, h1, accs[2 * k]);
            accs[2 * k + 1] = dot8w(wup, h0, h1, accs[2 * k + 1]);
        }
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) acc[rr] = warp_sum(acc[rr]);
#pragma unroll
    for (int k = 0; k < 2 * NSW; ++k) accs[k] = warp_sum(accs[k]);
    if (lane == 0) {
        float a[2 + NSW];
        int idx[2 + NSW];
        a[0] = silu(acc[0]) * acc[2];
        a[1] = silu(acc[1]) * acc[3];
        idx[0] = 2 * warp;
        idx[1] = 2 * warp + 1;
#pragma unroll
        for (int k = 0; k < NSW; ++k) {
            a[2 + k] = silu(accs[2 * k]) * accs[2 * k + 1];
            idx[2 + k] = 16 + k * 8 + warp;
        }
#pragma unroll
        for (int k = 0; k < 2 + NSW; ++k) {
            if (f16_out_of_range(a[k])) atomicOr(p.status, QW_DEV_RANGE);
            sact[idx[k]] = __half2float(__float2half_rn(a[k]));  // the activation is stored as fp16
        }
    }
    __syncthreads();
    trace_at(tr, 4);
    // ---- split-K down_proj: outputs 4t .. 4t+3 over this CTA's NA inputs ---------------
    float4 pp = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < NA; ++i) {
        const uint2 w = *reinterpret_cast<const uint2*>(wd_s + i * D1_D + 4 * t);
        const float a = sact[i];
        pp.x = fmaf(bf_lo(w.x), a, pp.x);
        pp.y = fmaf(bf_hi(w.x), a, pp.y);
        pp.z = fmaf(bf_lo(w.y), a, pp.z);
        pp.w = fmaf(bf_hi(w.y), a, pp.w);
    }
    // reduce-scatter: outputs 4t .. 4t+3 belong to CTA t / 32, which adds the 8 ranks'
    // slices of its rows [128 r, 128 r + 128) in order of rank
    cluster_wait();  // every CTA's mbarrier is initialised
    trace_at(tr, 5);
    st_async_f4(su32(rbuf + rank * D1_ROWS_M + 4 * (t & 31)), su32(&bar_r), (uint32_t)(t >> 5), pp);
    if (!mbar_wait0(&bar_r) && t == 0) atomicOr(p.status, QW_DEV_TIMEOUT);
    trace_at(tr, 6);
    if (t < D1_ROWS_M) {
        float s = 0.f;
#pragma unroll
        for (int r = 0; r < D1_CLM; ++r) s += rbuf[r * D1_ROWS_M + t];
        // clusters 2k and 2k + 1 meet in slot k, zeroed beforehand: 0 + a + b = a + b in
        // either order (two addends), so the sum does not depend on which lands first
        atomicAdd(p.dpart + (size_t)(c >> 1) * D1_D + D1_ROWS_M * rank + t, s);
    }
    trace_at(tr, 7);
}

// x + sum_c part[c] (in order of c) into out: the hidden state after a layer of this path,
// for the per-layer debug dump.
__global__ void k_dec1_sum(const float* __restrict__ x, const float* __restrict__ part, int n, int D,
                           float* __restrict__ out) {
    pdl_launch();
    pdl_wait();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < D; i += gridDim.x * blockDim.x) {
        float v = x[i];
        for (int c = 0; c < n; ++c) v += part[(size_t)c * D + i];
        out[i] = v;
    }
}

// dst[z][c][r] = src[z][r][c] for z < batch (rows, cols multiples of 32)
__global__ void k_transpose_bf16(const bf16* __restrict__ src, int rows, int cols, bf16* __restrict__ dst) {
    __shared__ bf16 tile[32][33];
    const size_t z = blockIdx.z;
    src += z * rows * cols;
    dst += z * rows * cols;
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    for (int i = threadIdx.y; i < 32; i += 8) tile[i][threadIdx.x] = src[(size_t)(r0 + i) * cols + c0 + threadIdx.x];
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += 8) dst[(size_t)(c0 + i) * rows + r0 + threadIdx.x] = tile[threadIdx.x][i];
}

namespace {

template <typename K>
bool dec1_attrs(K* k, int smem) {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess &&
           cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
}

template <typename K>
int dec1_clusters(K* k, int grid, int smem, int cl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(D1_THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = cl;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

template <int NA>
bool mlp_ready() {
    static int state = 0;  // 0 unknown, 1 ready, -1 not available
    if (state == 0) {
        state = -1;
        if (dec1_attrs(k_dec1_mlp<NA>, mlp_smem<NA>()) &&
            dec1_clusters(k_dec1_mlp<NA>, D1_NB * D1_CLM, mlp_smem<NA>(), D1_CLM) >= D1_NB)
            state = 1;
    }
    return state == 1;
}

bool attn_ready(int n_kv) {
    static int clusters = -1;
    if (clusters < 0) {
        clusters = 0;
        if (dec1_attrs(k_dec1_attn, A_SMEM)) clusters = dec1_clusters(k_dec1_attn, D1_CL, A_SMEM, D1_CL);
    }
    return clusters >= n_kv;
}

template <int NA>
cudaError_t mlp_go(const LaunchCtx& c, const Dec1Mlp& p) {
    if (!mlp_ready<NA>()) return cudaErrorNotSupported;
    return launch_kc(c, k_dec1_mlp<NA>, dim3(D1_NB * D1_CLM), dim3(D1_THREADS), (size_t)mlp_smem<NA>(), D1_CLM, p);
}

}  // namespace

int dec1_max_keys() { return D1_MAXPG * 16; }
int dec1_parts() { return D1_NP; }

bool dec1_available(int D, int I, int QD, int n_heads, int n_kv) {
    if (D != D1_D || QD != n_heads * 128 || n_heads != 2 * n_kv || n_kv < 1 || n_kv > 8) return false;
    bool mlp = false;
    switch (I) {
        case 128 * 16: mlp = mlp_ready<16>(); break;
        case 128 * 24: mlp = mlp_ready<24>(); break;
        case 128 * 32: mlp = mlp_ready<32>(); break;
        default: return false;
    }
    return mlp && attn_ready(n_kv);
}

cudaError_t launch_dec1_attn(const LaunchCtx& c, const Dec1Attn& p) {
    if (!attn_ready(p.n_kv)) return cudaErrorNotSupported;
    return launch_kc(c, k_dec1_attn, dim3(p.n_kv * D1_CL), dim3(D1_THREADS), (size_t)A_SMEM, D1_CL, p);
}

cudaError_t launch_dec1_mlp(const LaunchCtx& c, const Dec1Mlp& p) {
    switch (p.I) {
        case 128 * 16: return mlp_go<16>(c, p);
        case 128 * 24: return mlp_go<24>(c, p);
        case 128 * 32: return mlp_go<32>(c, p);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_dec1_sum(const LaunchCtx& c, const float* x, const float* part, int n, int D, float* out) {
    return launch_k(c, k_dec1_sum, dim3((D + 255) / 256), dim3(256), 0, x, part, n, D, out);
}

cudaError_t launch_transpose_bf16(cudaStream_t st, const bf16* src, int rows, int cols, int batch, bf16* dst) {
    if (rows % 32 || cols % 32 || batch < 1) return cudaErrorInvalidValue;
    k_transpose_bf16<<<dim3(cols / 32, rows / 32, batch), dim3(32, 8), 0, st>>>(src, rows, cols, dst);
    return cudaGetLastError();
}
