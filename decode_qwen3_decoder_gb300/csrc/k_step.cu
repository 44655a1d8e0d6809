// Batched decode step of the Qwen3-style decoder ("Dentro de un LLM: Inferencia en Python
// puro para Qwen3-0.6B en MLX", Pasos 5-7 for every layer) as ONE cooperative launch, for
// decode steps of 16-64 sequences (one new token each).
//
// Why: at batch 64 a step reads 1.19 GB of weights and ~8 GB of cached K/V. The K/V reads
// are pure bandwidth, but the four projections of a layer are a chain of small dependent
// matrix products (4-13 MB of weights each) whose cost is latency, not bytes. Sequences are
// independent, so the batch is split into two halves (A, B): while one half's attention
// streams its K/V, the other half runs its projection chain. Here both run inside one
// kernel, on disjoint CTAs, ordered by counters in global memory instead of kernel
// boundaries:
//
//  * CTAs [0, gp) -- projection role. Each phase (q|k|v, o_proj, gate/up, down_proj of one
//    layer and half) is a set of units = (128-row weight tile, K range); unit u of phase i
//    belongs to CTA (u + 13 i) mod gp. A producer warp streams the weight k-blocks of the
//    CTA's units, in program order, through an 11-stage TMA ring (128 x 64 fp16, 128-byte
//    swizzle): weights depend on nothing computed in the step, so the ring runs ahead across
//    phases and layers while the CTA waits for activations. Per unit, once its inputs are
//    complete, one thread loads the token operand (32 rows of the half, K range of the unit)
//    with TMA from an fp16 activation buffer, one thread issues tcgen05.mma (M = 128 weight
//    rows, N = 32 tokens, fp16, fp32 accumulator in TMEM), and four warps write the fp32
//    partial to global memory. The last unit of a tile to arrive (an atomic ticket) adds the
//    K-range partials in a fixed order and applies the epilogue:
//      q|k|v     x RMSNorm scale of the token, QK-norm + RoPE + KV append, q stored;
//      gate/up   x RMSNorm scale, SiLU(gate) * up stored;
//      o / down  x += W h, the token's sums of squares per 128-feature block, and
//                fp16(x * w) for the next RMSNorm (w = its weight): the next q|k|v or
//                gate/up operand, whose 1/RMS is applied in that epilogue (RMSNorm is a
//                per-token scale, so it commutes with the projection).
//    It then bumps the phase's completion counter.
//  * CTAs [gp, grid) -- attention role. Eight warps each take (token, KV head, key range)
//    units of each layer and half and run a flash-decode online softmax over the cached
//    16-key pages for both query heads of the KV head; each warp streams its pages (K and V,
//    4 KB each) with bulk TMA copies into its own 3-stage ring. Key ranges merge in the warp
//    that finishes last.
//
// Dependencies (per layer l and half h): all q|k|v tiles -> attention of (., g) -> o_proj
// units of K range g -> gate/up -> down_proj units of K range s (act features of gate/up
// tiles [6s, 6s + 6)) -> q|k|v of layer l + 1. The projection program interleaves the halves
// (o, gate/up, down, next q|k|v of A; then of B) so that half B's chain runs while half A's
// attention runs and vice versa. Every unit waits only on units that come earlier in the
// other CTAs' programs, and all CTAs are co-resident (cooperative launch), so the waits end.
// Each wait is bounded: on timeout the kernel records QW_DEV_TIMEOUT, raises a global abort
// word that stops every CTA, lets its copies and MMAs complete, frees TMEM and returns.
//
// Cross-CTA data is read with ld.global.cg (L2) or TMA, never through the non-coherent path;
// producers publish with __threadfence() (and a generic-to-async proxy fence, since the
// consumers read with TMA) before their counter increments.
#include "qw_internal.h"
#include "tc_sm103.cuh"
#include "gemm_epi.cuh"

namespace {

constexpr int ST_THREADS = 256;
constexpr int ST_NST = 11;                               // weight ring stages
constexpr int ST_STAGE = BM * BK * 2;                    // one 128 x 64 fp16 k-block (16 KB)
constexpr int ST_MAXKB = 8;                              // k-blocks per unit
constexpr int ST_N = kStepMaxHalf;                       // MMA N: the 32 token rows of a half
constexpr int ST_BBOX = ST_N * 128;                      // one [32][64] fp16 operand box (4 KB)
constexpr int ST_BBYTES = ST_MAXKB * ST_BBOX;            // token operand (32 KB)
constexpr int A_NPS = 3;                                 // attention: page stages per warp
constexpr int A_STAGE = 2 * 16 * 128 * 2;                // K and V of one 16-key page (8 KB)
// shared memory (offsets from a 1024-aligned base). Projection role: weight ring, then the
// token operand, whose space the epilogue reuses for its staging tile. Attention role: one
// page ring per warp over the same space.
constexpr int SO_B = ST_NST * ST_STAGE;
constexpr int SO_END0 = SO_B + ST_BBYTES;
static_assert((ST_THREADS / 32) * A_NPS * A_STAGE <= SO_END0, "attention rings fit the projection space");
static_assert(32 * EP * 4 <= ST_BBYTES, "epilogue staging fits the operand space");
constexpr int SO_NW = SO_END0;
constexpr int SO_META = SO_NW + 256 * 4;
constexpr int SO_RED = SO_META + 64 * 4;
constexpr int SO_RS = SO_RED + 4 * 32 * 4;
constexpr int SO_BAR = SO_RS + 32 * 4;
constexpr int ST_NBAR = 2 * ST_NST + 3;  // full[], empty[], operand full, accumulator ready, MMA drain
constexpr int SO_ABAR = SO_BAR + ST_NBAR * 8;
constexpr int SO_MISC = SO_ABAR + (ST_THREADS / 32) * A_NPS * 8;
constexpr int ST_SMEM = 1024 + SO_MISC + 64;

enum { KQKV = 0, KO = 1, KGU = 2, KDN = 3 };
// completion-counter slots of one (layer, half)
constexpr int DS_QKV = 0;   // + KV head g: q|k|v tiles of g (target 4)
constexpr int DS_ATT = 16;  // + KV head g: merged (token, g) attention outputs (target: tokens)
constexpr int DS_O = 32;    // o_proj tiles (target D / 128)
constexpr int DS_GU = 33;   // + s: gate/up tiles of down_proj's K range s (target tiles / 8)
constexpr int DS_DN = 41;   // down_proj tiles (target D / 128)
constexpr int DS_QKV_ALL = 42;  // all q|k|v tiles (target QKVR / 128): what the attention CTAs wait for
constexpr int DN_SPLIT = 8;

struct Geo {
    int tiles, S, kb;  // 128-row weight tiles, K ranges, k-blocks per unit
};
__device__ __forceinline__ Geo geo(const StepKParams& p, int kind) {
    switch (kind) {
        case KQKV: return {p.QKVR / 128, 2, p.D / 128};
        case KO: return {p.D / 128, p.n_kv, p.QD / 64 / p.n_kv};
        case KGU: return {2 * p.I / 128, 2, p.D / 128};
        default: return {p.D / 128, DN_SPLIT, p.I / 64 / DN_SPLIT};
    }
}
// first partial slot / ticket of each kind within a half
__device__ __forceinline__ int unit_off(const StepKParams& p, int kind) {
    int o = 0;
    for (int k = 0; k < kind; ++k) {
        const Geo g = geo(p, k);
        o += g.tiles * g.S;
    }
    return o;
}
__device__ __forceinline__ int tile_off(const StepKParams& p, int kind) {
    int o = 0;
    for (int k = 0; k < kind; ++k) o += geo(p, k).tiles;
    return o;
}
// Phase i of the projection program: q|k|v of layer 0 for both halves, then per layer l and
// half h: o_proj, gate/up, down_proj of (l, h) and q|k|v of (l + 1, h).
__device__ __forceinline__ bool phase_at(const StepKParams& p, int i, int& kind, int& l, int& h) {
    if (i < 2) {
        kind = KQKV;
        l = 0;
        h = i;
        return true;
    }
    const int j = i - 2, r = j & 7, k = r & 3;
    l = j >> 3;
    h = r >> 2;
    kind = (k == 0) ? KO : (k == 1) ? KGU : (k == 2) ? KDN : KQKV;
    if (k == 3) {
        l += 1;
        if (l >= p.L) return false;
    }
    return true;
}
__device__ __forceinline__ int n_phases(const StepKParams& p) { return 2 + 8 * p.L; }
__device__ __forceinline__ int first_unit(int c, int i, int gp) { return ((c - 13 * i) % gp + gp) % gp; }

__device__ __forceinline__ int* done_ctr(const StepKParams& p, int l, int h, int slot) {
    return p.done + (((size_t)l * 2 + h) * kStepDoneSlots + slot) * kStepDoneStride;
}

__device__ __forceinline__ int ld_relaxed(const int* a) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}
__device__ __forceinline__ uint4 ldcg16(const void* a) { return __ldcg(reinterpret_cast<const uint4*>(a)); }
// generic-proxy global writes of this thread vs. later TMA reads (either side of a handoff)
__device__ __forceinline__ void fence_proxy_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
// Bounded wait that ignores the abort flags: used to let this CTA's own copies and MMAs land
// before it exits.
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > kTcWaitNs) return false;
    return true;
}

// Wait until *ctr >= target, bounded by p.wait_ns; gives up at once if the grid aborted. A
// timeout records QW_DEV_TIMEOUT and aborts the grid. The counter is polled with relaxed
// loads (a backoff keeps the line free for the increments); one fence orders what follows.
__device__ bool wait_ge(const StepKParams& p, const int* ctr, int target) {
    if (ld_relaxed(ctr) >= target) {
        __threadfence();
        return true;
    }
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        __nanosleep(n < 4 ? 64 : 256);
        if (ld_relaxed(ctr) >= target) {
            __threadfence();
            return true;
        }
        if ((n & 15u) == 0) {
            if (*(volatile int*)p.abort_g) return false;
            if (globaltimer_ns() - t0 > p.wait_ns) {
                atomicOr(p.status, QW_DEV_TIMEOUT);
                atomicExch(p.abort_g, 1);
                return false;
            }
        }
    }
}

// Trace record k of CTA c (8 words): id, then up to seven %globaltimer stamps.
__device__ __forceinline__ void trace_rec(const StepKParams& p, int k, unsigned long long id, uint64_t a, uint64_t b,
                                          uint64_t c2, uint64_t d, uint64_t e = 0, uint64_t f = 0, uint64_t g = 0) {
    if (!p.trace || k >= p.trace_n) return;
    unsigned long long* r = p.trace + ((size_t)blockIdx.x * p.trace_n + k) * 8;
    r[0] = id;
    r[1] = a;
    r[2] = b;
    r[3] = c2;
    r[4] = d;
    r[5] = e;
    r[6] = f;
    r[7] = g;
}

// ---- attention role -------------------------------------------------------------------

__device__ __forceinline__ float dot8(const float* q, const uint4 k) {
    float a = q[0] * h_lo(k.x);
    a = fmaf(q[1], h_hi(k.x), a);
    a = fmaf(q[2], h_lo(k.y), a);
    a = fmaf(q[3], h_hi(k.y), a);
    a = fmaf(q[4], h_lo(k.z), a);
    a = fmaf(q[5], h_hi(k.z), a);
    a = fmaf(q[6], h_lo(k.w), a);
    a = fmaf(q[7], h_hi(k.w), a);
    return a;
}
__device__ __forceinline__ float hsum16(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    return v;
}

struct WarpSoftmax {
    float q0[8], q1[8];  // the two query heads' dims [dl, dl + 8), scaled to the exp2 domain
    float m0, m1, l0, l1;
    float o0[8], o1[8];
};

// One page of 16 keys (this lane: keys 2i + half, dims [dl, dl + 8)): scores, running max,
// rescale and P V. Slots at or past nvalid get zero weight and zero values.
__device__ __forceinline__ void page_step(WarpSoftmax& w, const uint4 (&kk)[8], uint4 (&vv)[8], int nvalid, int half) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (2 * i + half >= nvalid) vv[i] = make_uint4(0u, 0u, 0u, 0u);
    float s0[8], s1[8];
    float pm0 = -INFINITY, pm1 = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float d0 = hsum16(dot8(w.q0, kk[i]));
        const float d1 = hsum16(dot8(w.q1, kk[i]));
        const bool valid = (2 * i + half) < nvalid;
        s0[i] = valid ? d0 : -INFINITY;
        s1[i] = valid ? d1 : -INFINITY;
        pm0 = fmaxf(pm0, s0[i]);
        pm1 = fmaxf(pm1, s1[i]);
    }
    pm0 = fmaxf(pm0, __shfl_xor_sync(0xffffffffu, pm0, 16));
    pm1 = fmaxf(pm1, __shfl_xor_sync(0xffffffffu, pm1, 16));
    const float n0 = fmaxf(w.m0, pm0), n1 = fmaxf(w.m1, pm1);
    if (n0 == -INFINITY) return;  // nothing valid yet (n1 is then -inf too)
    const float a0 = exp2f(w.m0 - n0), a1 = exp2f(w.m1 - n1);
    w.m0 = n0;
    w.m1 = n1;
    w.l0 *= a0;
    w.l1 *= a1;
#pragma unroll
    for (int d = 0; d < 8; ++d) {
        w.o0[d] *= a0;
        w.o1[d] *= a1;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float e0 = exp2f(s0[i] - w.m0), e1 = exp2f(s1[i] - w.m1);
        w.l0 += e0;
        w.l1 += e1;
        const uint32_t vw[4] = {vv[i].x, vv[i].y, vv[i].z, vv[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float va = h_lo(vw[j]), vb = h_hi(vw[j]);
            w.o0[2 * j] = fmaf(e0, va, w.o0[2 * j]);
            w.o0[2 * j + 1] = fmaf(e0, vb, w.o0[2 * j + 1]);
            w.o1[2 * j] = fmaf(e1, va, w.o1[2 * j]);
            w.o1[2 * j + 1] = fmaf(e1, vb, w.o1[2 * j + 1]);
        }
    }
}

// Attention of token `tok` (query heads 2g, 2g+1 over KV head g), keys [k0, k1), by one warp.
// The warp's pages stream through its ring (A_NPS stages at `ring`, barriers from `bar0`);
// pc counts the pages this warp has streamed (it sets each stage's phase).
__device__ void attn_unit(const StepKParams& p, int l, int h, int tok, int g, int s, int n_act, int k0, int k1,
                          uint8_t* ring, uint32_t bar0, uint32_t& pc) {
    const int lane = threadIdx.x & 31, half = lane >> 4, dl = (lane & 15) * 8;
    WarpSoftmax w;
    {
        const f16* qp = p.q + (size_t)tok * p.QD + (size_t)(2 * g) * 128 + dl;
        const uint4 a = ldcg16(qp), b = ldcg16(qp + 128);
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            w.q0[2 * i] = h_lo(aw[i]) * p.scale_log2;
            w.q0[2 * i + 1] = h_hi(aw[i]) * p.scale_log2;
            w.q1[2 * i] = h_lo(bw[i]) * p.scale_log2;
            w.q1[2 * i + 1] = h_hi(bw[i]) * p.scale_log2;
        }
    }
    w.m0 = w.m1 = -INFINITY;
    w.l0 = w.l1 = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) w.o0[i] = w.o1[i] = 0.f;
    const int seq = p.tv.seq[tok];
    const int* pt = p.kv.page_table + (size_t)seq * p.kv.max_pages_per_seq;
    const f16* Kl = p.kv.k + (size_t)l * p.kv.layer_stride;
    const f16* Vl = p.kv.v + (size_t)l * p.kv.layer_stride;
    const int p0 = k0 >> 4, np = ((k1 + 15) >> 4) - p0;
    // page ids of the first 32 pages of the range, one per lane (one load for all of them)
    const int pt_lane = (lane < np) ? pt[p0 + lane] : -1;
    auto page_of = [&](int i) {  // called by all lanes
        const int pid = (i < 32) ? __shfl_sync(0xffffffffu, pt_lane, i & 31) : pt[p0 + i];
        return (pid < 0 || pid >= p.kv.n_pages) ? -1 : pid;  // a missing page is reported by the append
    };
    auto issue = [&](int i) {  // called by all lanes; lane 0 copies page i into its stage
        const int pid = page_of(i);
        if (lane == 0) {
            const uint32_t k = pc + (uint32_t)i, st = k % A_NPS;
            const uint32_t bar = bar0 + 8 * st;
            const size_t off = ((size_t)(pid < 0 ? 0 : pid) * p.n_kv + g) * 16 * 128;
            mbar_expect_tx(bar, A_STAGE);
            bulk_g2s(smem_u32(ring + st * A_STAGE), Kl + off, A_STAGE / 2, bar);
            bulk_g2s(smem_u32(ring + st * A_STAGE + A_STAGE / 2), Vl + off, A_STAGE / 2, bar);
        }
    };
    for (int i = 0; i < np && i < A_NPS; ++i) issue(i);
    for (int i = 0; i < np; ++i) {
        const uint32_t k = pc + (uint32_t)i, st = k % A_NPS;
        if (!mbar_drain(bar0 + 8 * st, (k / A_NPS) & 1u) && lane == 0) atomicOr(p.status, QW_DEV_TIMEOUT);
        const uint8_t* pk = ring + st * A_STAGE;
        uint4 kk[8], vv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            kk[j] = *reinterpret_cast<const uint4*>(pk + ((2 * j + half) * 128 + dl) * 2);
            vv[j] = *reinterpret_cast<const uint4*>(pk + A_STAGE / 2 + ((2 * j + half) * 128 + dl) * 2);
        }
        const int nvalid = page_of(i) < 0 ? 0 : min(16, k1 - (p0 + i) * 16);
        page_step(w, kk, vv, nvalid, half);
        __syncwarp();
        if (i + A_NPS < np) issue(i + A_NPS);
    }
    pc += (uint32_t)np;
    // the two half-warps saw alternate keys with the same running max
    w.l0 += __shfl_xor_sync(0xffffffffu, w.l0, 16);
    w.l1 += __shfl_xor_sync(0xffffffffu, w.l1, 16);
#pragma unroll
    for (int d = 0; d < 8; ++d) {
        w.o0[d] += __shfl_xor_sync(0xffffffffu, w.o0[d], 16);
        w.o1[d] += __shfl_xor_sync(0xffffffffu, w.o1[d], 16);
    }
    // lanes 0-15 hold head 2g, lanes 16-31 head 2g + 1, dims [dl, dl + 8)
    const float* oo = half ? w.o1 : w.o0;
    const float mm = half ? w.m1 : w.m0, ll = half ? w.l1 : w.l0;
    const int head = 2 * g + half;
    f16* outp = p.attn + (size_t)tok * p.QD + (size_t)head * 128 + dl;
    f16* dbgp = p.dbg_attn ? p.dbg_attn + ((size_t)l * p.T + tok) * p.QD + (size_t)head * 128 + dl : nullptr;
    auto store8 = [&](const float* v, float inv) {
        uint4 u;
        u.x = pack_h2(v[0] * inv, v[1] * inv);
        u.y = pack_h2(v[2] * inv, v[3] * inv);
        u.z = pack_h2(v[4] * inv, v[5] * inv);
        u.w = pack_h2(v[6] * inv, v[7] * inv);
        *reinterpret_cast<uint4*>(outp) = u;
        if (dbgp) *reinterpret_cast<uint4*>(dbgp) = u;
    };
    int* att_done = done_ctr(p, l, h, DS_ATT + g);
    if (n_act == 1) {
        store8(oo, 1.0f / ll);
        fence_proxy_global();
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(att_done, 1);
        return;
    }
    const size_t slot = ((size_t)tok * p.n_heads + head) * p.att_stride + s;
    float4* po = reinterpret_cast<float4*>(p.att_po + slot * 128 + dl);
    __stcg(po, make_float4(oo[0], oo[1], oo[2], oo[3]));
    __stcg(po + 1, make_float4(oo[4], oo[5], oo[6], oo[7]));
    if ((lane & 15) == 0) __stcg(reinterpret_cast<float2*>(p.att_pml + slot * 2), make_float2(mm, ll));
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) last = (atomicAdd(p.att_cnt + (size_t)tok * p.n_kv + g, 1) == n_act - 1);
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();
    const size_t base = ((size_t)tok * p.n_heads + head) * p.att_stride;
    // the splits' maxima: lane j of each half-warp holds split j (16 per round)
    float M = -INFINITY;
    for (int j0 = 0; j0 < n_act; j0 += 16) {
        const int j = j0 + (lane & 15);
        const float mj = __ldcg(p.att_pml + (base + min(j, n_act - 1)) * 2);
        M = fmaxf(M, j < n_act ? mj : -INFINITY);
    }
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 8));
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 4));
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 2));
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 1));
    float L = 0.f, A[8];
#pragma unroll
    for (int d = 0; d < 8; ++d) A[d] = 0.f;
    for (int j0 = 0; j0 < n_act; j0 += 4) {  // four splits' loads in flight, added in order
        float2 ml[4];
        float4 x0[4], x1[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const size_t jj = base + min(j0 + r, n_act - 1);
            ml[r] = __ldcg(reinterpret_cast<const float2*>(p.att_pml + jj * 2));
            const float4* pj = reinterpret_cast<const float4*>(p.att_po + jj * 128 + dl);
            x0[r] = __ldcg(pj);
            x1[r] = __ldcg(pj + 1);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            if (j0 + r < n_act) {
                const float f = exp2f(ml[r].x - M);
                L += ml[r].y * f;
                A[0] += x0[r].x * f; A[1] += x0[r].y * f; A[2] += x0[r].z * f; A[3] += x0[r].w * f;
                A[4] += x1[r].x * f; A[5] += x1[r].y * f; A[6] += x1[r].z * f; A[7] += x1[r].w * f;
            }
        }
    }
    store8(A, 1.0f / L);
    if (lane == 0) p.att_cnt[(size_t)tok * p.n_kv + g] = 0;
    fence_proxy_global();
    __threadfence();
    __syncwarp();
    if (lane == 0) atomicAdd(att_done, 1);
}

}  // namespace

__global__ void __launch_bounds__(ST_THREADS, 1) k_step(const __grid_constant__ StepMaps mp, const __grid_constant__ StepKParams p) {
    extern __shared__ uint8_t st_smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(st_smem_raw) + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;

    if (c >= p.gp) {
        // ---------------- attention role ----------------
        const int aw = (c - p.gp) * (ST_THREADS / 32) + warp;
        const int naw = ((int)gridDim.x - p.gp) * (ST_THREADS / 32);
        uint8_t* ring = smem + warp * A_NPS * A_STAGE;
        const uint32_t bar0 = smem_u32(smem + SO_ABAR + warp * A_NPS * 8);
        volatile int* a_ok = reinterpret_cast<volatile int*>(smem + SO_MISC);
        if (lane == 0) {
            for (int i = 0; i < A_NPS; ++i) mbar_init(bar0 + 8 * i, 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncwarp();
        uint32_t pc = 0;
        int nrec = 0;
        for (int l = 0; l < p.L; ++l) {
            for (int h = 0; h < 2; ++h) {
                // one thread per CTA waits for every q|k|v tile of (l, h); the warps follow
                const uint64_t tw = p.trace ? globaltimer_ns() : 0;
                if (threadIdx.x == 0) *a_ok = wait_ge(p, done_ctr(p, l, h, DS_QKV_ALL), p.QKVR / 128) ? 1 : 0;
                __syncthreads();
                const int go = *a_ok;
                __syncthreads();  // read by all before thread 0 can write the next phase's flag
                if (!go) return;  // nothing of this warp is in flight between phases
                if (lane == 0) fence_proxy_global();  // this warp's copies read what the q|k|v epilogues wrote
                const uint64_t ts = p.trace ? globaltimer_ns() : 0;
                const int nh = p.nh[h];
                const int U = nh * p.n_kv * p.nsplit;
                for (int u = aw; u < U; u += naw) {
                    const int t = u / (p.n_kv * p.nsplit);
                    const int g = (u / p.nsplit) % p.n_kv;
                    const int s = u % p.nsplit;
                    const int tok = p.t0[h] + t;
                    const int n_keys = p.tv.pos[tok] + 1;
                    const int n_act = (n_keys + p.chunk - 1) / p.chunk;
                    if (s >= n_act) continue;
                    const uint64_t tu = p.trace ? globaltimer_ns() : 0;
                    attn_unit(p, l, h, tok, g, s, n_act, s * p.chunk, min((s + 1) * p.chunk, n_keys), ring, bar0, pc);
                    if (p.trace && warp == 0 && lane == 0)
                        trace_rec(p, nrec++, (1ull << 40) | ((unsigned long long)l << 24) | ((unsigned long long)h << 20) | u,
                                  tw, ts, tu, globaltimer_ns());
                }
            }
        }
        return;
    }

    // ---------------- projection role ----------------
    uint8_t* ring = smem;
    uint8_t* Bop = smem + SO_B;
    float* E = reinterpret_cast<float*>(smem + SO_B);  // epilogue staging over the operand space
    float* nws = reinterpret_cast<float*>(smem + SO_NW);
    int* tpos = reinterpret_cast<int*>(smem + SO_META);
    int* tdst = tpos + 32;
    float* red = reinterpret_cast<float*>(smem + SO_RED);
    float* s_rs = reinterpret_cast<float*>(smem + SO_RS);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + SO_BAR);
    uint64_t* empty = full + ST_NST;
    uint64_t* bfull = empty + ST_NST;
    uint64_t* accf = bfull + 1;
    uint64_t* mdrain = accf + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SO_MISC);
    volatile int* abort_s = reinterpret_cast<volatile int*>(smem + SO_MISC + 4);
    volatile int* s_flag = reinterpret_cast<volatile int*>(smem + SO_MISC + 8);

    if (threadIdx.x == 0) {
        for (int s = 0; s < ST_NST; ++s) {
            mbar_init(smem_u32(full + s), 1);
            mbar_init(smem_u32(empty + s), 1);
        }
        mbar_init(smem_u32(bfull), 1);
        mbar_init(smem_u32(accf), 1);
        mbar_init(smem_u32(mdrain), 1);
        *abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 4 && lane == 0) {
        for (int i = 0; i < 4; ++i) tma_prefetch_desc(&mp.w[i]);
        tma_prefetch_desc(&mp.xw);
        tma_prefetch_desc(&mp.attn);
        tma_prefetch_desc(&mp.act);
    }
    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(32)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int gp = p.gp;
    const int NP = n_phases(p);

    if (warp == 4) {
        // ---- producer: the weight k-blocks of this CTA's units, in program order ----
        if (lane == 0) {
            uint32_t rc = 0;
            bool ok = true;
            for (int i = 0; i < NP && ok; ++i) {
                int kind, l, h;
                if (!phase_at(p, i, kind, l, h)) continue;
                const Geo G = geo(p, kind);
                const CUtensorMap* map = &mp.w[kind];
                const int rows_per_layer = kind == KQKV ? p.QKVR : kind == KGU ? 2 * p.I : p.D;
                for (int u = first_unit(c, i, gp); u < G.tiles * G.S && ok; u += gp) {
                    const int tile = u / G.S, split = u % G.S;
                    for (int j = 0; j < G.kb; ++j) {
                        const int s = rc % ST_NST;
                        const uint32_t ph = (rc / ST_NST) & 1u;
                        if (!mbar_wait(smem_u32(empty + s), ph ^ 1u, abort_s)) {
                            *abort_s = 1;
                            ok = false;
                            break;
                        }
                        mbar_expect_tx(smem_u32(full + s), ST_STAGE);
                        tma_load_2d(smem_u32(ring + s * ST_STAGE), map, smem_u32(full + s), (split * G.kb + j) * BK,
                                    l * rows_per_layer + tile * BM);
                        ++rc;
                    }
                }
            }
            // let every copy this CTA issued land before the CTA can exit
            for (uint32_t r = (rc > ST_NST ? rc - ST_NST : 0); r < rc; ++r)
                mbar_drain(smem_u32(full + r % ST_NST), (r / ST_NST) & 1u);
        }
        __syncwarp();
    } else if (warp == 5) {
        // ---- MMA issuer ----
        if (lane == 0) {
            uint32_t rc = 0, uc = 0;
            bool ok = true, issued = false;
            constexpr uint32_t idesc = idesc_f16(BM, ST_N);
            for (int i = 0; i < NP && ok; ++i) {
                int kind, l, h;
                if (!phase_at(p, i, kind, l, h)) continue;
                const Geo G = geo(p, kind);
                for (int u = first_unit(c, i, gp); u < G.tiles * G.S && ok; u += gp) {
                    if (!mbar_wait(smem_u32(bfull), uc & 1u, abort_s)) {
                        *abort_s = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int j = 0; j < G.kb; ++j) {
                        const int s = rc % ST_NST;
                        const uint32_t ph = (rc / ST_NST) & 1u;
                        if (!mbar_wait(smem_u32(full + s), ph, abort_s)) {
                            *abort_s = 1;
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t ad = sw128_desc(smem_u32(ring + s * ST_STAGE));
                        const uint64_t bd = sw128_desc(smem_u32(Bop + j * ST_BBOX));
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)
                            umma_f16(tmem, ad + 2 * k, bd + 2 * k, idesc, (j > 0 || k > 0) ? 1u : 0u);
                        umma_commit(smem_u32(empty + s));
                        issued = true;
                        ++rc;
                    }
                    if (!ok) break;
                    umma_commit(smem_u32(accf));
                    ++uc;
                }
            }
            if (issued) {  // every MMA of this CTA has completed before TMEM is freed
                umma_commit(smem_u32(mdrain));
                mbar_drain(smem_u32(mdrain), 0u);
            }
        }
        __syncwarp();
    } else if (warp < 4) {
        // ---- operand loads + epilogue (threads 0-127 = TMEM lanes = tile rows) ----
        const int tid = threadIdx.x;
        uint32_t uc = 0, bc = 0;
        bool ok = true;
        int nrec = 0;
        uint64_t tr0 = 0, tr1 = 0, tr2 = 0;
        for (int i = 0; i < NP && ok; ++i) {
            int kind, l, h;
            if (!phase_at(p, i, kind, l, h)) continue;
            const Geo G = geo(p, kind);
            const int nh = p.nh[h], tok0 = p.t0[h];
            const int UT = unit_off(p, 4);
            const CUtensorMap* bmap = (kind == KO) ? &mp.attn : (kind == KDN) ? &mp.act : &mp.xw;
            for (int u = first_unit(c, i, gp); u < G.tiles * G.S; u += gp) {
                const int tile = u / G.S, split = u % G.S;
                // 1. wait for this unit's inputs, then load its token operand with TMA
                if (tid == 0 && p.trace) tr0 = globaltimer_ns();
                if (tid == 0) {
                    const int* ctr = nullptr;
                    int target = 0;
                    if (kind == KQKV) {
                        if (l > 0) {
                            ctr = done_ctr(p, l - 1, h, DS_DN);
                            target = p.D / 128;
                        }
                    } else if (kind == KO) {
                        ctr = done_ctr(p, l, h, DS_ATT + split);
                        target = nh + ((l == 0 && h == 0 && split == 0) ? p.extra : 0);
                    } else if (kind == KGU) {
                        ctr = done_ctr(p, l, h, DS_O);
                        target = p.D / 128;
                    } else {
                        ctr = done_ctr(p, l, h, DS_GU + split);
                        target = geo(p, KGU).tiles / DN_SPLIT;
                    }
                    const bool good = (ctr == nullptr || wait_ge(p, ctr, target));
                    *s_flag = good ? 1 : 0;
                    if (good) {
                        fence_proxy_global();  // the copies read what other CTAs' epilogues wrote
                        mbar_expect_tx(smem_u32(bfull), G.kb * ST_BBOX);
                        for (int j = 0; j < G.kb; ++j)
                            tma_load_2d(smem_u32(Bop + j * ST_BBOX), bmap, smem_u32(bfull), (split * G.kb + j) * BK, tok0);
                        ++bc;
                    }
                }
                named_bar_epi();
                if (!*s_flag) {
                    ok = false;
                    break;
                }
                if (tid == 0 && p.trace) tr1 = globaltimer_ns();
                // the RMSNorm scale of each token (q|k|v, gate/up) from its per-block sums of squares
                if ((kind == KQKV || kind == KGU) && tid < nh) {
                    const float* sp = p.ss + (size_t)(tok0 + tid) * (p.D / 128);
                    float acc = 0.f;
                    for (int b = 0; b < p.D / 128; ++b) acc += __ldcg(sp + b);
                    s_rs[tid] = rsqrtf(acc / (float)p.D + p.eps);
                }
                // 2. accumulator -> fp32 partial of this K range ([row][token], this thread's row)
                if (!mbar_wait(smem_u32(accf), uc & 1u, abort_s)) {
                    *abort_s = 1;
                    ok = false;
                    break;
                }
                ++uc;
                if (tid == 0 && p.trace) tr2 = globaltimer_ns();
                tc_fence_after();
                uint32_t r[32];
                TMEM_LD32(tmem + ((uint32_t)(warp * 32) << 16), r);
                tmem_wait_ld();
                tc_fence_before();
                int* tick = p.tick + h * tile_off(p, 4) + tile_off(p, kind) + tile;
                float v[32];
                {
                    float4* part_u = reinterpret_cast<float4*>(p.part + (((size_t)h * UT + unit_off(p, kind) + u) * 128 + tid) * 32);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        __stcg(part_u + q, make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                                       __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3])));
                    __threadfence();
                    named_bar_epi();
                    if (tid == 0) *s_flag = (atomicAdd(tick, 1) == G.S - 1) ? 1 : 0;
                    named_bar_epi();
                    if (!*s_flag) {
                        if (tid == 0) trace_rec(p, nrec++, ((unsigned long long)i << 16) | u, tr0, tr1, tr2, globaltimer_ns());
                        continue;
                    }
                    // 3. last K range of the tile: add the partials in order, two at a time
                    __threadfence();
#pragma unroll
                    for (int t = 0; t < 32; ++t) v[t] = 0.f;
                    const float4* pt0 = reinterpret_cast<const float4*>(
                        p.part + (((size_t)h * UT + unit_off(p, kind) + tile * G.S) * 128 + tid) * 32);
                    for (int s2 = 0; s2 < G.S; s2 += 2) {
                        float4 a[8], b[8];
                        const int s3 = min(s2 + 1, G.S - 1);
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            a[q] = __ldcg(pt0 + (size_t)s2 * 128 * 8 + q);
                            b[q] = __ldcg(pt0 + (size_t)s3 * 128 * 8 + q);
                        }
                        const bool two = s2 + 1 < G.S;
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            v[4 * q] += a[q].x;
                            v[4 * q + 1] += a[q].y;
                            v[4 * q + 2] += a[q].z;
                            v[4 * q + 3] += a[q].w;
                            if (two) {
                                v[4 * q] += b[q].x;
                                v[4 * q + 1] += b[q].y;
                                v[4 * q + 2] += b[q].z;
                                v[4 * q + 3] += b[q].w;
                            }
                        }
                    }
                }
                const uint64_t tr3 = (tid == 0 && p.trace) ? globaltimer_ns() : 0;
                int done_slot;
                if (kind == KO || kind == KDN) {
                    const int m = tile * BM + tid;
                    // the next RMSNorm's weight: post-attention of layer l, or input of layer l + 1
                    const bf16* wn = (kind == KO) ? p.norms + (size_t)l * (2 * p.D + 256) + p.D
                                     : (l + 1 < p.L) ? p.norms + (size_t)(l + 1) * (2 * p.D + 256)
                                                     : nullptr;
                    const float wm = wn ? __bfloat162float(wn[m]) : 0.f;
                    float xo[32];
#pragma unroll
                    for (int t = 0; t < 32; ++t) xo[t] = __ldcg(p.x + (size_t)(tok0 + min(t, nh - 1)) * p.D + m);
                    bool big = false;
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        if (t < nh) {
                            const float xn = xo[t] + v[t];
                            __stcg(p.x + (size_t)(tok0 + t) * p.D + m, xn);
                            v[t] = xn;
                            if (wn) {
                                const float y = xn * wm;
                                big |= f16_out_of_range(y);
                                p.xw[(size_t)(tok0 + t) * p.D + m] = __float2half_rn(y);
                            }
                            if (kind == KDN && p.dbg_hidden) p.dbg_hidden[((size_t)l * p.T + tok0 + t) * p.D + m] = xn;
                        }
                    }
                    if (big) atomicOr(p.status, QW_DEV_RANGE);
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        if (t < nh) {
                            const float q = warp_sum(v[t] * v[t]);
                            if (lane == 0) red[warp * 32 + t] = q;
                        }
                    }
                    named_bar_epi();
                    if (tid < nh)
                        __stcg(p.ss + (size_t)(tok0 + tid) * (p.D / 128) + tile,
                               red[tid] + red[32 + tid] + red[64 + tid] + red[96 + tid]);
                    done_slot = kind == KO ? DS_O : DS_DN;
                } else if (kind == KGU) {
#pragma unroll
                    for (int t = 0; t < 32; ++t) E[t * EP + tid] = v[t] * s_rs[t < nh ? t : 0];
                    named_bar_epi();
                    GemmKParams gk = {};
                    gk.out_h = p.act;
                    gk.ld_out = p.I;
                    gk.status = p.status;
                    epi_silu(gk, E, tok0, nh, tile);
                    done_slot = DS_GU + tile / (G.tiles / DN_SPLIT);
                } else {
                    f16* EH = reinterpret_cast<f16*>(E);
#pragma unroll
                    for (int t = 0; t < 32; ++t) EH[t * EPH + tid] = __float2half_rn(v[t] * s_rs[t < nh ? t : 0]);
                    GemmKParams gk = {};
                    const bf16* nb = p.norms + (size_t)l * (2 * p.D + 256);
                    gk.q_out = p.q;
                    gk.q_norm = nb + 2 * p.D;
                    gk.k_norm = nb + 2 * p.D + 128;
                    gk.eps = p.eps;
                    gk.rope_cos = p.rope_cos;
                    gk.rope_sin = p.rope_sin;
                    gk.tv = p.tv;
                    gk.kv = p.kv;
                    gk.layer = l;
                    gk.n_heads = p.n_heads;
                    gk.n_kv = p.n_kv;
                    gk.T = tok0 + nh;
                    gk.status = p.status;
                    gk.dbg_pos = l == 0 ? p.dbg_pos : nullptr;
                    gk.dbg_slot = l == 0 ? p.dbg_slot : nullptr;
                    load_norm_weights(gk, nws);
                    fill_tok_meta<32>(gk, tok0, tile, tpos, tdst);
                    named_bar_epi();
                    RopeRegs rr;
                    if (tile < p.n_heads + p.n_kv) load_rope(gk, tpos, 0, nh, rr);
                    epi_heads(gk, EH, nws, tdst, rr, tok0, 0, nh, tile);
                    const int g = tile < p.n_heads ? tile / 2 : tile < p.n_heads + p.n_kv ? tile - p.n_heads
                                                                                          : tile - p.n_heads - p.n_kv;
                    done_slot = DS_QKV + g;
                }
                const uint64_t tr4 = (tid == 0 && p.trace) ? globaltimer_ns() : 0;
                fence_proxy_global();
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // staging before the next operand copy
                __threadfence();
                named_bar_epi();
                if (tid == 0) {
                    *tick = 0;
                    __threadfence();
                    atomicAdd(done_ctr(p, l, h, done_slot), 1);
                    if (kind == KQKV) atomicAdd(done_ctr(p, l, h, DS_QKV_ALL), 1);
                    trace_rec(p, nrec++, (1ull << 39) | ((unsigned long long)i << 16) | u, tr0, tr1, tr2, globaltimer_ns(),
                              tr3, tr4, 0);
                }
            }
        }
        if (!ok) *abort_s = 1;
        // a token operand copy whose unit was abandoned must land before the CTA exits
        if (tid == 0 && bc > uc) mbar_drain(smem_u32(bfull), (bc - 1) & 1u);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(32) : "memory");
    }
}

// ---- host side --------------------------------------------------------------------------

bool step_shape_ok(int D, int I, int QD, int QKVR, int n_heads, int n_kv) {
    return D % 128 == 0 && D / 128 <= ST_MAXKB && D / 128 <= 16 && I % 512 == 0 && I / 64 / DN_SPLIT <= ST_MAXKB &&
           n_heads == 2 * n_kv && n_kv <= 16 && QD == n_heads * 128 && QKVR == QD + 2 * n_kv * 128 &&
           2 * I / 128 / DN_SPLIT >= 1 && QD / 64 / n_kv <= ST_MAXKB;
}

int step_tiles(int D, int I, int QKVR) { return QKVR / 128 + D / 128 + 2 * I / 128 + D / 128; }

size_t step_part_floats(int D, int I, int QKVR, int n_kv) {
    const size_t units = (size_t)(QKVR / 128) * 2 + (size_t)(D / 128) * n_kv + (size_t)(2 * I / 128) * 2 +
                         (size_t)(D / 128) * DN_SPLIT;
    return 2 * units * 32 * 128;
}

int step_smem_bytes() { return ST_SMEM; }

int step_blocks_per_sm() {
    if (cudaFuncSetAttribute(k_step, cudaFuncAttributeMaxDynamicSharedMemorySize, ST_SMEM) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_step, ST_THREADS, ST_SMEM) != cudaSuccess) return 0;
    return n;
}

cudaError_t launch_decode_step(cudaStream_t st, const StepKParams& p, const StepMaps& maps, int grid) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_step, cudaFuncAttributeMaxDynamicSharedMemorySize, ST_SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(ST_THREADS);
    cfg.dynamicSmemBytes = ST_SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_step, maps, p);
}
