// Persistent decode kernel: one whole decode step (<= 8 sequences, one new token each) of
// the Qwen3-style decoder ("Dentro de un LLM: Inferencia en Python puro para Qwen3-0.6B en
// MLX", Pasos 2-9) in a single cooperative launch with one CTA per SM.
//
// Why: at batch 1 a step reads 1.19 GB of weights but is a chain of ~140 dependent matrix
// products of 4-13 MB each; as separate launches every link pays launch and HBM-latency
// costs. Here the weight stream is decoupled from the dependency chain:
//
//  * the last warp (12) of every CTA is a producer: it walks the CTA's slice of every weight matrix
//    of the step in order (layer by layer: q|k|v, o_proj, gate+up, down_proj; then the LM
//    head) and streams it with cp.async.bulk (TMA) into a 7-stage shared-memory ring. The
//    weights depend on nothing computed in the step, so the producer runs up to 7 stages
//    ahead, across phase and layer boundaries, while the consumers wait on activations.
//  * warps 0-11 consume: after a grid barrier that publishes the previous phase's output,
//    they stage the activation rows in shared memory (RMSNorm fused for the q|k|v,
//    gate/up and LM-head inputs) and reduce each weight row of the ring against them.
//  * the attention phase (teams of 4 warps, one (token, KV head, key split) unit per team)
//    applies QK-norm + RoPE to the two query heads and the key of its KV head, appends the
//    new K/V to the paged cache, and runs an online softmax over the cached pages; splits
//    merge in the team that finishes last.
//  * the LM-head phase keeps a packed per-token argmax; the last CTA to finish writes the
//    greedy ids and advances the sequence lengths.
//
// Phases per layer: q|k|v -> attention -> o_proj(+residual) -> gate/up(+SiLU*mul) ->
// down_proj(+residual), each ended by a grid barrier. All waits are bounded (about 2 s):
// on timeout the kernel sets QW_DEV_TIMEOUT and an abort word that makes every CTA stop.
//
// Activations written and read within the kernel go through L2 (ld/st.cg), never the
// non-coherent read-only path.
#include <utility>

#include "qw_internal.h"

namespace {

constexpr int MK_CONS_WARPS = 12;  // one per work item of a stage
constexpr int MK_CONS_THREADS = MK_CONS_WARPS * 32;
constexpr int MK_PRODUCER_WARP = MK_CONS_WARPS;
constexpr int MK_THREADS = MK_CONS_THREADS + 32;
constexpr int MK_STAGE = 24 * 1024;
constexpr int MK_NST = 7;
constexpr int MK_ACT = 48 * 1024;
constexpr int MK_TEAMS = 3;  // attention teams of 4 warps
constexpr int MK_SEG = 1024;  // columns per work item
constexpr int MK_ITEMS = MK_STAGE / (MK_SEG * 2);  // work items per ring stage (12)
constexpr int MK_TMAX = 4;    // tokens per step
constexpr unsigned long long kMkWaitNs = 2000000000ull;

enum { PH_QKV = 0, PH_O = 1, PH_GU = 2, PH_D = 3, PH_LM = 4 };

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mb_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mb_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mb_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mb_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ int ld_acquire_i(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned ld_acquire_u(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Bounded wait on an mbarrier phase; gives up after ~2 s or when the kernel aborted.
__device__ bool mb_wait(uint32_t bar, uint32_t parity, const int* abort_g) {
    if (mb_try(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    uint32_t n = 0;
    while (true) {
        if (mb_try(bar, parity)) return true;
        if ((++n & 127u) == 0) {
            if (ld_acquire_i(abort_g)) return false;
            if (globaltimer_ns() - t0 > kMkWaitNs) return false;
        }
    }
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ uint4 ldg_nc4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr));
    return r;
}
__device__ __forceinline__ float4 lds128f(uint32_t addr) {
    float4 r;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "r"(addr));
    return r;
}
// 8 bf16 weights (widened exactly by a shift) against 8 fp32 activations
__device__ __forceinline__ float dot8b(const uint4 w, const float4 a0, const float4 a1, float acc) {
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
__device__ __forceinline__ float half16_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    return v;
}

}  // namespace



namespace {

struct Slice {
    const bf16* a;
    const bf16* b;
    int r0, n, K, rs;
};

__device__ __forceinline__ Slice slice_of(const MkParams& p, int kind, int l, int c, int G) {
    Slice s;
    int N;
    s.b = nullptr;
    switch (kind) {
        case PH_QKV: N = p.QKV; s.K = p.D; s.a = p.wqkv + (size_t)l * p.QKV * p.D; break;
        case PH_O: N = p.D; s.K = p.QD; s.a = p.wo + (size_t)l * p.D * p.QD; break;
        case PH_GU:
            N = p.I; s.K = p.D;
            s.a = p.wg + (size_t)l * p.I * p.D;
            s.b = p.wu + (size_t)l * p.I * p.D;
            break;
        case PH_D: N = p.D; s.K = p.I; s.a = p.wd + (size_t)l * p.D * p.I; break;
        default: N = p.V; s.K = p.D; s.a = p.embed; break;
    }
    s.r0 = (int)((long long)N * c / G);
    s.n = (int)((long long)N * (c + 1) / G) - s.r0;
    // rows per stage: 12 work items of MK_SEG columns (gate and up rows count as two items)
    s.rs = (kind == PH_GU) ? MK_ITEMS / 2 : MK_ITEMS / (s.K / MK_SEG);
    return s;
}

// Grid barrier among the consumer warps of all CTAs. The arrival counter only grows within
// a step: barrier k of the step completes when it reaches G * (k + 1). Thread 0 publishes
// its CTA's writes with one release-add and polls the counter with acquire loads (no
// fences, no read-modify-write on the critical path). A failure seen by any warp of the
// CTA (my_ok false) turns into an abort of the whole grid. Returns false on abort.
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ bool grid_sync(const MkParams& p, unsigned G, unsigned k, bool my_ok, volatile int* s_fail,
                          volatile int* s_ok) {
    if (!my_ok) *s_fail = 1;
    named_sync(1, MK_CONS_THREADS);
    if (threadIdx.x == 0) {
        int ok = (*s_fail == 0);
        if (p.trace && k < (unsigned)p.trace_n) p.trace[(size_t)blockIdx.x * 8 * p.trace_n + 2 * k] = globaltimer_ns();
        if (!ok) {
            atomicExch(p.abort_g, 1);
        } else {
            red_release_add(p.sync, 1u);
            const unsigned target = G * (k + 1);
            const uint64_t t0 = globaltimer_ns();
            uint32_t n = 0;
            while (ld_acquire_u(p.sync) < target) {
                if ((++n & 31u) == 0) {
                    if (ld_acquire_i(p.abort_g)) {
                        ok = 0;
                        break;
                    }
                    if (globaltimer_ns() - t0 > kMkWaitNs) {
                        atomicOr(p.status, QW_DEV_TIMEOUT);
                        atomicExch(p.abort_g, 1);
                        ok = 0;
                        break;
                    }
                }
            }
        }
        *s_ok = ok;
        if (p.trace && k < (unsigned)p.trace_n) p.trace[(size_t)blockIdx.x * 8 * p.trace_n + 2 * k + 1] = globaltimer_ns();
    }
    named_sync(1, MK_CONS_THREADS);
    return *s_ok != 0;
}

}  // namespace

__global__ void __launch_bounds__(MK_THREADS, 1) k_decode_mk(const MkParams p) {
    extern __shared__ uint8_t mk_smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(mk_smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* ring = smem;
    uint8_t* actb = smem + MK_NST * MK_STAGE;  // activation rows / attention team scratch
    uint64_t* full = reinterpret_cast<uint64_t*>(actb + MK_ACT);
    uint64_t* empty = full + MK_NST;
    __shared__ float s_red[MK_CONS_WARPS][MK_TMAX];  // per-warp sums of squares of the staged rows
    __shared__ unsigned long long s_best[MK_CONS_WARPS][MK_TMAX];
    __shared__ int s_last;
    __shared__ volatile uint32_t s_issued;
    __shared__ volatile int s_fail;
    __shared__ volatile int s_ok;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned G = gridDim.x;
    const int c = blockIdx.x;
    const int T = p.T;

    if (threadIdx.x == 0) {
        s_issued = 0;
        s_fail = 0;
        for (int i = 0; i < MK_NST; ++i) {
            mb_init(su32(full + i), 1);
            mb_init(su32(empty + i), 1);  // released once per stage, after the stage barrier
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    // ===================================== producer =====================================
    if (warp == MK_PRODUCER_WARP) {
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int l = 0; l <= p.n_layers && ok; ++l) {
                const int k0 = (l < p.n_layers) ? PH_QKV : PH_LM, k1 = (l < p.n_layers) ? PH_D : PH_LM;
                for (int kind = k0; kind <= k1 && ok; ++kind) {
                    const Slice sl = slice_of(p, kind, l, c, G);
                    const uint32_t rb = (uint32_t)sl.K * 2u;
                    for (int j = 0; j < sl.n; j += sl.rs, ++it) {
                        const int nr = min(sl.rs, sl.n - j);
                        const int st = it % MK_NST;
                        const uint32_t ph = (it / MK_NST) & 1u;
                        if (!mb_wait(su32(empty + st), ph ^ 1u, p.abort_g)) {
                            ok = false;
                            break;
                        }
                        const uint32_t dst = su32(ring + st * MK_STAGE);
                        const uint32_t bytes = (uint32_t)nr * rb;
                        mb_expect_tx(su32(full + st), sl.b ? 2u * bytes : bytes);
                        bulk_g2s(dst, sl.a + (size_t)(sl.r0 + j) * sl.K, bytes, su32(full + st));
                        if (sl.b) bulk_g2s(dst + bytes, sl.b + (size_t)(sl.r0 + j) * sl.K, bytes, su32(full + st));
                        s_issued = it + 1;
                        if (p.trace && it < 2u * p.trace_n)
                            p.trace[(size_t)c * 8 * p.trace_n + 6 * p.trace_n + it] = globaltimer_ns();
                    }
                }
            }
            if (!ok) {
                atomicOr(p.status, QW_DEV_TIMEOUT);
                atomicExch(p.abort_g, 1);
            }
        }
        return;
    }

    // ===================================== consumers ====================================
    uint32_t it = 0;
    bool ok = true;
    float* hs = reinterpret_cast<float*>(actb);  // fp32 activation rows [T][K]
    const uint32_t hs_addr = su32(hs);
    __shared__ float s_part[2][MK_ITEMS][MK_TMAX];

    unsigned nbar = 0;  // grid barriers passed in this step
    auto gsync = [&](bool mine) -> bool { return grid_sync(p, G, nbar++, mine, &s_fail, &s_ok); };

    // Weights of one phase. Each ring stage holds 12 work items of MK_SEG columns (row
    // segments; a gate row and an up row are separate items). Warp w < 12 reduces item w
    // against the staged activations with four independent chains per token; the partial
    // sums meet in shared memory and, after a CTA barrier, warp r combines the items of
    // row r in fixed order (deterministic) and calls out(row, value[t]) from lane t.
    auto consume = [&](int kind, int l, auto&& out) -> bool {
        const Slice sl = slice_of(p, kind, l, c, G);
        const int S = (kind == PH_GU) ? 1 : sl.K / MK_SEG;
        const uint32_t rb = (uint32_t)sl.K * 2u;
        bool good = true;
        for (int j = 0; j < sl.n; j += sl.rs, ++it) {
            const int nr = min(sl.rs, sl.n - j);
            const int items = (kind == PH_GU) ? 2 * nr : nr * S;
            const int st = it % MK_NST;
            const uint32_t ph = (it / MK_NST) & 1u;
            const bool tr = p.trace && warp == 0 && lane == 0 && it < 2u * p.trace_n;
            if (tr) p.trace[(size_t)c * 8 * p.trace_n + 2 * p.trace_n + 2 * it] = globaltimer_ns();
            if (good && !mb_wait(su32(full + st), ph, p.abort_g)) {
                good = false;
                if (lane == 0) {
                    atomicOr(p.status, QW_DEV_TIMEOUT);
                    atomicExch(p.abort_g, 1);
                }
            }
            if (tr) p.trace[(size_t)c * 8 * p.trace_n + 2 * p.trace_n + 2 * it + 1] = globaltimer_ns();
            float (*part)[MK_TMAX] = s_part[it & 1u];
            if (good && warp < items) {
                uint32_t wa, aa;
                const uint32_t st_addr = su32(ring + st * MK_STAGE);
                if (kind == PH_GU) {
                    wa = st_addr + ((warp & 1) * nr + (warp >> 1)) * rb;
                    aa = hs_addr;
                } else {
                    wa = st_addr + (warp / S) * rb + (warp % S) * (MK_SEG * 2);
                    aa = hs_addr + (warp % S) * (MK_SEG * 4);
                }
                uint4 w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) w[q] = lds128(wa + (q * 256 + lane * 8) * 2);
                float acc[MK_TMAX][4];
#pragma unroll
                for (int t = 0; t < MK_TMAX; ++t) {
                    if (t < T) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint32_t ap = aa + (uint32_t)(t * sl.K + q * 256 + lane * 8) * 4u;
                            acc[t][q] = dot8b(w[q], lds128f(ap), lds128f(ap + 16), 0.f);
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < MK_TMAX; ++t) {
                    if (t < T) {
                        const float v = warp_sum((acc[t][0] + acc[t][1]) + (acc[t][2] + acc[t][3]));
                        if (lane == t) part[warp][t] = v;
                    }
                }
            }
            named_sync(5, MK_CONS_THREADS);
            if (warp == 0 && lane == 0) mb_arrive(su32(empty + st));  // the stage's data is consumed
            if (good && warp < nr && lane < T) {
                float v[2];
                if (kind == PH_GU) {
                    v[0] = part[2 * warp][lane];
                    v[1] = part[2 * warp + 1][lane];
                } else {
                    float a = 0.f;
                    for (int q = 0; q < S; ++q) a += part[warp * S + q][lane];
                    v[0] = a;
                    v[1] = 0.f;
                }
                out(sl.r0 + j + warp, lane, v);
            }
        }
        return good;
    };

    // RMSNorm input of the T residual rows (Paso 3) in one pass: x * w (w = the norm weight)
    // into fp32 shared memory while each warp sums its tokens' squares (s_red). 1/RMS is a
    // per-token scale, so the consumers apply it to the reduced products (rs_of).
    auto stage_norm = [&](const bf16* w) {
        float ssp[MK_TMAX];
#pragma unroll
        for (int t = 0; t < MK_TMAX; ++t) ssp[t] = 0.f;
        for (int i = threadIdx.x; i < T * p.D / 4; i += MK_CONS_THREADS) {
            const int t = i / (p.D / 4), k = (i % (p.D / 4)) * 4;
            const float4 v = __ldcg(reinterpret_cast<const float4*>(p.x) + i);
            const uint2 wb = *reinterpret_cast<const uint2*>(w + k);
            const float q = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
#pragma unroll
            for (int u = 0; u < MK_TMAX; ++u)
                if (u == t) ssp[u] += q;
            *reinterpret_cast<float4*>(hs + i * 4) =
                make_float4(v.x * bf_lo(wb.x), v.y * bf_hi(wb.x), v.z * bf_lo(wb.y), v.w * bf_hi(wb.y));
        }
#pragma unroll
        for (int t = 0; t < MK_TMAX; ++t) {
            const float q = warp_sum(ssp[t]);
            if (lane == 0) s_red[warp][t] = q;
        }
        named_sync(1, MK_CONS_THREADS);
    };
    // 1/RMS of token t from the per-warp sums of squares (fixed order)
    auto rs_of = [&](int t) {
        float q = 0.f;
#pragma unroll
        for (int w = 0; w < MK_CONS_WARPS; ++w) q += s_red[w][t];
        return rsqrtf(q / (float)p.D + p.eps);
    };

    // Weights of one layer phase: the CTA's slice is at most MK_NST ring stages, all issued
    // ahead by the producer. Every warp reduces work items across all of those stages at once,
    // then one CTA barrier releases the stages, and the rows' sums (items added in fixed
    // order) go out. More stages than the ring are taken in batches.
    __shared__ float s_part2[2][MK_NST * MK_ITEMS][MK_TMAX];
    auto consume_all = [&](int kind, int l, bool normed, auto&& out) -> bool {
        const Slice sl = slice_of(p, kind, l, c, G);
        const int S = (kind == PH_GU) ? 1 : sl.K / MK_SEG;  // items per row (gate and up: one each)
        const int ipr = (kind == PH_GU) ? 2 : S;
        const uint32_t rb = (uint32_t)sl.K * 2u;
        const int n_st = (sl.n + sl.rs - 1) / sl.rs;
        bool good = true;
        for (int b0 = 0; b0 < n_st; b0 += MK_NST) {
            const int nb = min(MK_NST, n_st - b0);
            const int rows_b = min(sl.n - b0 * sl.rs, nb * sl.rs);
            const int items_b = rows_b * ipr;  // stages hold MK_ITEMS items each but the last
            float (*part)[MK_TMAX] = s_part2[(it + b0) & 1u];
            for (int item = warp; item < items_b && good; item += MK_CONS_WARPS) {
                const int sb = item / MK_ITEMS, ii = item % MK_ITEMS;
                const uint32_t k = it + b0 + sb;
                const int st = k % MK_NST;
                const int nr = min(sl.rs, rows_b - sb * sl.rs);  // rows in this stage
                if (!mb_wait(su32(full + st), (k / MK_NST) & 1u, p.abort_g)) {
                    good = false;
                    if (lane == 0) {
                        atomicOr(p.status, QW_DEV_TIMEOUT);
                        atomicExch(p.abort_g, 1);
                    }
                    break;
                }
                uint32_t wa, aa;
                const uint32_t st_addr = su32(ring + st * MK_STAGE);
                if (kind == PH_GU) {
                    wa = st_addr + ((ii & 1) * nr + (ii >> 1)) * rb;
                    aa = hs_addr;
                } else {
                    wa = st_addr + (ii / S) * rb + (ii % S) * (MK_SEG * 2);
                    aa = hs_addr + (ii % S) * (MK_SEG * 4);
                }
                uint4 wv[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) wv[q] = lds128(wa + (q * 256 + lane * 8) * 2);
                float acc[MK_TMAX][4];
#pragma unroll
                for (int t = 0; t < MK_TMAX; ++t) {
                    if (t < T) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint32_t ap = aa + (uint32_t)(t * sl.K + q * 256 + lane * 8) * 4u;
                            acc[t][q] = dot8b(wv[q], lds128f(ap), lds128f(ap + 16), 0.f);
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < MK_TMAX; ++t) {
                    if (t < T) {
                        const float v = warp_sum((acc[t][0] + acc[t][1]) + (acc[t][2] + acc[t][3]));
                        if (lane == t) part[item][t] = v;
                    }
                }
            }
            if (!good) s_fail = 1;
            named_sync(5, MK_CONS_THREADS);
            if (warp == 0 && lane < nb) mb_arrive(su32(empty + (it + b0 + lane) % MK_NST));  // stages consumed
            good = good && (s_fail == 0);
            if (good) {
                for (int r = warp; r < rows_b; r += MK_CONS_WARPS) {
                    if (lane < T) {
                        const int base = (r / sl.rs) * MK_ITEMS + (r % sl.rs) * ipr;
                        float v[2];
                        if (kind == PH_GU) {
                            v[0] = part[base][lane];
                            v[1] = part[base + 1][lane];
                        } else {
                            float a = 0.f;
                            for (int q = 0; q < S; ++q) a += part[base + q][lane];
                            v[0] = a;
                            v[1] = 0.f;
                        }
                        if (normed) {
                            const float rs = rs_of(lane);
                            v[0] *= rs;
                            v[1] *= rs;
                        }
                        out(sl.r0 + b0 * sl.rs + r, lane, v);
                    }
                }
            }
        }
        it += (uint32_t)n_st;
        return good;
    };
    // fp16 activation rows [T][K] (through L2) widened into fp32 shared memory.
    auto stage_h = [&](const f16* src, int K) {
        for (int i = threadIdx.x; i < T * K / 8; i += MK_CONS_THREADS) {
            const uint4 a = __ldcg(reinterpret_cast<const uint4*>(src) + i);
            *reinterpret_cast<float4*>(hs + i * 8) = make_float4(h_lo(a.x), h_hi(a.x), h_lo(a.y), h_hi(a.y));
            *reinterpret_cast<float4*>(hs + i * 8 + 4) = make_float4(h_lo(a.z), h_hi(a.z), h_lo(a.w), h_hi(a.w));
        }
        named_sync(1, MK_CONS_THREADS);
    };
    // Warm L2 with the cached K/V pages this CTA's attention units will read in layer l
    // (at most 8 pages per unit: the latency of the first loads is what matters).
    auto prefetch_kv = [&](int l) {
        if (warp >= MK_TEAMS || lane != 0) return;
        const int units = T * p.n_kv * p.n_splits;
        for (int u = c + G * warp; u < units; u += G * MK_TEAMS) {
            const int t = u / (p.n_kv * p.n_splits), g = (u / p.n_splits) % p.n_kv, s = u % p.n_splits;
            const int seq = p.seq[t];
            const int n_keys = p.kv.len[seq];  // cached keys (the new one is written later)
            const int k0 = s * p.chunk, k1 = min(k0 + p.chunk, n_keys);
            const int* pt = p.kv.page_table + (size_t)seq * p.kv.max_pages_per_seq;
            for (int pg = k0 >> 4, n = 0; pg < ((k1 + 15) >> 4) && n < 8; ++pg, ++n) {
                const int page = pt[pg];
                if (page < 0 || page >= p.kv.n_pages) continue;
                const size_t off = ((size_t)page * p.n_kv + g) * 16 * 128;
                const f16* kp = p.kv.k + (size_t)l * p.kv.layer_stride + off;
                const f16* vp = p.kv.v + (size_t)l * p.kv.layer_stride + off;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(kp), "r"(16 * 128 * 2) : "memory");
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(vp), "r"(16 * 128 * 2) : "memory");
            }
        }
    };

    // ---- phase 0: embedding gather (Paso 2) -------------------------------------------
    {
        const int total = T * p.D / 4;
        const int per = (total + G - 1) / G;
        for (int i = c * per + threadIdx.x; i < min(total, (c + 1) * per); i += MK_CONS_THREADS) {
            const int t = i / (p.D / 4), k = (i % (p.D / 4)) * 4;
            const int id = p.ids[t];
            const bool bad = id < 0 || id >= p.V;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
            if (!bad) {
                const uint2 wv = *reinterpret_cast<const uint2*>(p.embed + (size_t)id * p.D + k);
                o = make_float4(bf_lo(wv.x), bf_hi(wv.x), bf_lo(wv.y), bf_hi(wv.y));
            } else if (k == 0) {
                atomicOr(p.status, QW_DEV_BAD_TOKEN);
            }
            __stcg(reinterpret_cast<float4*>(p.x + (size_t)t * p.D + k), o);
        }
        ok = gsync(true);
    }

    for (int l = 0; l < p.n_layers && ok; ++l) {
        const bf16* nb = p.norms + (size_t)l * (2 * p.D + 256);
        // ---- q|k|v projections (Paso 5), input RMSNorm fused -------------------------
        prefetch_kv(l);
        stage_norm(nb);
        ok = consume_all(PH_QKV, l, true, [&](int row, int t, const float* v) { __stcg(p.qkv + (size_t)t * p.QKV + row, v[0]); });
        if (!(ok = gsync(ok))) break;

        // ---- attention (Paso 5): QK-norm, RoPE, KV append, split-KV online softmax -----
        {
            const int team = warp >> 2, wt = warp & 3;
            if (team < MK_TEAMS) {
                float* sq = reinterpret_cast<float*>(actb) + team * 1408;          // [2][128]
                float* so = sq + 256;                                             // [4][2][128]
                float* sm = so + 1024;                                            // [4][2] max
                float* sl_ = sm + 8;                                              // [4][2] sum
                int* slast = reinterpret_cast<int*>(sl_ + 8);
                const int units = T * p.n_kv * p.n_splits;
                const int bar_id = 2 + team;
                const int NH = p.n_heads + 2 * p.n_kv;
                const f16* Kl = p.kv.k + (size_t)l * p.kv.layer_stride;
                const f16* Vl = p.kv.v + (size_t)l * p.kv.layer_stride;
                for (int u = c + G * team; u < units; u += G * MK_TEAMS) {
                    const int t = u / (p.n_kv * p.n_splits);
                    const int g = (u / p.n_splits) % p.n_kv;
                    const int s = u % p.n_splits;
                    const int seq = p.seq[t];
                    const int pos = p.kv.len[seq];
                    const int n_keys = pos + 1;
                    const int n_act = (n_keys + p.chunk - 1) / p.chunk;
                    if (s >= n_act) continue;
                    const int* pt = p.kv.page_table + (size_t)seq * p.kv.max_pages_per_seq;
                    const bool writer = (s == n_act - 1);
                    // QK-norm + RoPE of q heads 2g, 2g+1 and k head g; v copied
                    {
                        const int hh_ = wt < 2 ? 2 * g + wt : (wt == 2 ? p.n_heads + g : p.n_heads + p.n_kv + g);
                        const float4 xv = __ldcg(reinterpret_cast<const float4*>(p.qkv + (size_t)t * NH * 128 + hh_ * 128 + lane * 4));
                        float y[4] = {xv.x, xv.y, xv.z, xv.w};
                        if (wt < 3) {
                            const bf16* nw = nb + 2 * p.D + (wt < 2 ? 0 : 128);
                            const float ss = warp_sum(y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3]);
                            const float r = rsqrtf(ss * (1.0f / 128.0f) + p.eps);
                            const uint2 wb = *reinterpret_cast<const uint2*>(nw + lane * 4);
                            y[0] *= r * bf_lo(wb.x);
                            y[1] *= r * bf_hi(wb.x);
                            y[2] *= r * bf_lo(wb.y);
                            y[3] *= r * bf_hi(wb.y);
                            const int i0 = (lane & 15) * 4;
                            const float4 cs = *reinterpret_cast<const float4*>(p.rcos + (size_t)pos * 64 + i0);
                            const float4 sn = *reinterpret_cast<const float4*>(p.rsin + (size_t)pos * 64 + i0);
                            const float cc[4] = {cs.x, cs.y, cs.z, cs.w}, sv[4] = {sn.x, sn.y, sn.z, sn.w};
                            float o4[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float pj = __shfl_xor_sync(0xffffffffu, y[j], 16);
                                o4[j] = (lane < 16) ? (y[j] * cc[j] - pj * sv[j]) : (pj * sv[j] + y[j] * cc[j]);
                            }
#pragma unroll
                            for (int j = 0; j < 4; ++j) y[j] = o4[j];
                        }
                        if (wt < 2) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) sq[wt * 128 + lane * 4 + j] = y[j];
                        } else if (writer) {
                            const int pi = pos >> 4;
                            const int page = (pi < p.kv.max_pages_per_seq) ? pt[pi] : -1;
                            if (page < 0 || page >= p.kv.n_pages) {
                                if (lane == 0) atomicOr(p.status, QW_DEV_BAD_POS);
                            } else {
                                f16* pool = (wt == 2 ? p.kv.k : p.kv.v) + (size_t)l * p.kv.layer_stride;
                                if (f16_out_of_range(y[0]) || f16_out_of_range(y[1]) || f16_out_of_range(y[2]) ||
                                    f16_out_of_range(y[3]))
                                    atomicOr(p.status, QW_DEV_RANGE);
                                uint2 pk;
                                pk.x = pack_h2(y[0], y[1]);
                                pk.y = pack_h2(y[2], y[3]);
                                *reinterpret_cast<uint2*>(pool + (((size_t)page * p.n_kv + g) * 16 + (pos & 15)) * 128 + lane * 4) = pk;
                                if (l == 0 && p.dbg_pos && wt == 2 && g == 0 && lane == 0) {
                                    p.dbg_pos[t] = pos;
                                    p.dbg_slot[t] = page * 16 + (pos & 15);
                                }
                            }
                        }
                    }
                    named_sync(bar_id, 128);
                    const int half = lane >> 4, dl = (lane & 15) * 8;
                    float q0[8], q1[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        q0[i] = sq[dl + i] * p.scale_log2;
                        q1[i] = sq[128 + dl + i] * p.scale_log2;
                    }
                    const int k0 = s * p.chunk, k1 = min(k0 + p.chunk, n_keys);
                    const int p0 = k0 >> 4, p1 = (k1 + 15) >> 4;
                    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, o0[8], o1[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) o0[i] = o1[i] = 0.f;
                    for (int pg = p0 + wt; pg < p1; pg += 4) {
                        const int page = pt[pg];
                        if (page < 0 || page >= p.kv.n_pages) continue;
                        const int nvalid = min(16, k1 - pg * 16);
                        const size_t off = ((size_t)page * p.n_kv + g) * 16 * 128 + dl;
                        uint4 kr[8], vr[8];
                        if (writer && pg == p1 - 1) {
#pragma unroll
                            for (int i = 0; i < 8; ++i) kr[i] = *reinterpret_cast<const uint4*>(Kl + off + (size_t)(2 * i + half) * 128);
#pragma unroll
                            for (int i = 0; i < 8; ++i) vr[i] = *reinterpret_cast<const uint4*>(Vl + off + (size_t)(2 * i + half) * 128);
                        } else {
#pragma unroll
                            for (int i = 0; i < 8; ++i) kr[i] = ldg_nc4(Kl + off + (size_t)(2 * i + half) * 128);
#pragma unroll
                            for (int i = 0; i < 8; ++i) vr[i] = ldg_nc4(Vl + off + (size_t)(2 * i + half) * 128);
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            if (2 * i + half >= nvalid) vr[i] = make_uint4(0u, 0u, 0u, 0u);
                        float s0[8], s1[8], pm0 = -INFINITY, pm1 = -INFINITY;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            float d0 = 0.f, d1 = 0.f;
                            const uint32_t kw[4] = {kr[i].x, kr[i].y, kr[i].z, kr[i].w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                d0 = fmaf(q0[2 * j], h_lo(kw[j]), d0);
                                d0 = fmaf(q0[2 * j + 1], h_hi(kw[j]), d0);
                                d1 = fmaf(q1[2 * j], h_lo(kw[j]), d1);
                                d1 = fmaf(q1[2 * j + 1], h_hi(kw[j]), d1);
                            }
                            d0 = half16_sum(d0);
                            d1 = half16_sum(d1);
                            const bool valid = (2 * i + half) < nvalid;
                            s0[i] = valid ? d0 : -INFINITY;
                            s1[i] = valid ? d1 : -INFINITY;
                            pm0 = fmaxf(pm0, s0[i]);
                            pm1 = fmaxf(pm1, s1[i]);
                        }
                        pm0 = fmaxf(pm0, __shfl_xor_sync(0xffffffffu, pm0, 16));
                        pm1 = fmaxf(pm1, __shfl_xor_sync(0xffffffffu, pm1, 16));
                        const float n0 = fmaxf(m0, pm0), n1 = fmaxf(m1, pm1);
                        const float a0 = exp2f(m0 - n0), a1 = exp2f(m1 - n1);
                        m0 = n0;
                        m1 = n1;
                        l0 *= a0;
                        l1 *= a1;
#pragma unroll
                        for (int d = 0; d < 8; ++d) {
                            o0[d] *= a0;
                            o1[d] *= a1;
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float e0 = exp2f(s0[i] - m0), e1 = exp2f(s1[i] - m1);
                            l0 += e0;
                            l1 += e1;
                            const uint32_t vw[4] = {vr[i].x, vr[i].y, vr[i].z, vr[i].w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float va = h_lo(vw[j]), vb = h_hi(vw[j]);
                                o0[2 * j] = fmaf(e0, va, o0[2 * j]);
                                o0[2 * j + 1] = fmaf(e0, vb, o0[2 * j + 1]);
                                o1[2 * j] = fmaf(e1, va, o1[2 * j]);
                                o1[2 * j + 1] = fmaf(e1, vb, o1[2 * j + 1]);
                            }
                        }
                    }
                    l0 += __shfl_xor_sync(0xffffffffu, l0, 16);
                    l1 += __shfl_xor_sync(0xffffffffu, l1, 16);
#pragma unroll
                    for (int d = 0; d < 8; ++d) {
                        o0[d] += __shfl_xor_sync(0xffffffffu, o0[d], 16);
                        o1[d] += __shfl_xor_sync(0xffffffffu, o1[d], 16);
                    }
                    if (lane < 16) {
#pragma unroll
                        for (int d = 0; d < 8; ++d) {
                            so[(wt * 2 + 0) * 128 + dl + d] = o0[d];
                            so[(wt * 2 + 1) * 128 + dl + d] = o1[d];
                        }
                    }
                    if (lane == 0) {
                        sm[wt * 2] = m0;
                        sm[wt * 2 + 1] = m1;
                        sl_[wt * 2] = l0;
                        sl_[wt * 2 + 1] = l1;
                    }
                    named_sync(bar_id, 128);
                    const int tt = threadIdx.x & 127;
                    const int hh2 = tt >> 6, d2 = (tt & 63) * 2;
                    float M = -INFINITY;
#pragma unroll
                    for (int w = 0; w < 4; ++w) M = fmaxf(M, sm[w * 2 + hh2]);
                    float L = 0.f, O0 = 0.f, O1 = 0.f;
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float f = exp2f(sm[w * 2 + hh2] - M);
                        L += sl_[w * 2 + hh2] * f;
                        O0 += so[(w * 2 + hh2) * 128 + d2] * f;
                        O1 += so[(w * 2 + hh2) * 128 + d2 + 1] * f;
                    }
                    const int head = 2 * g + hh2;
                    f16* outp = p.o + ((size_t)t * p.n_heads + head) * 128 + d2;
                    if (n_act == 1) {
                        __stcg(reinterpret_cast<unsigned*>(outp), pack_h2(O0 / L, O1 / L));
                    } else {
                        const size_t slot = ((size_t)t * p.n_heads + head) * p.n_splits + s;
                        __stcg(reinterpret_cast<float2*>(p.part_o + slot * 128 + d2), make_float2(O0, O1));
                        if ((tt & 63) == 0) __stcg(reinterpret_cast<float2*>(p.part_ml + slot * 2), make_float2(M, L));
                        __threadfence();
                        named_sync(bar_id, 128);
                        if (tt == 0) {
                            const int ticket = atomicAdd(p.counters + (size_t)t * p.n_kv + g, 1);
                            *slast = (ticket == n_act - 1);
                        }
                        named_sync(bar_id, 128);
                        if (*slast) {
                            __threadfence();
                            const size_t base = ((size_t)t * p.n_heads + head) * p.n_splits;
                            float MM = -INFINITY;
                            for (int j = 0; j < n_act; ++j) MM = fmaxf(MM, __ldcg(p.part_ml + (base + j) * 2));
                            float LL = 0.f, A0 = 0.f, A1 = 0.f;
                            for (int j = 0; j < n_act; ++j) {
                                const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml + (base + j) * 2));
                                const float f = exp2f(ml.x - MM);
                                const float2 ov = __ldcg(reinterpret_cast<const float2*>(p.part_o + (base + j) * 128 + d2));
                                LL += ml.y * f;
                                A0 += ov.x * f;
                                A1 += ov.y * f;
                            }
                            __stcg(reinterpret_cast<unsigned*>(outp), pack_h2(A0 / LL, A1 / LL));
                            if (tt == 0) p.counters[(size_t)t * p.n_kv + g] = 0;
                        }
                    }
                    named_sync(bar_id, 128);  // team scratch is reused by the next unit
                }
            }
        }
        if (!(ok = gsync(true))) break;

        // ---- o_proj + residual (Pasos 5, 7) -------------------------------------------
        stage_h(p.o, p.QD);
        ok = consume_all(PH_O, l, false, [&](int row, int t, const float* v) {
            float* xp = p.x + (size_t)t * p.D + row;
            __stcg(xp, __ldcg(xp) + v[0]);
        });
        if (!(ok = gsync(ok))) break;

        // ---- gate/up + SiLU*mul (Paso 6), post-attention RMSNorm fused -----------------
        stage_norm(nb + p.D);
        ok = consume_all(PH_GU, l, true, [&](int row, int t, const float* v) {
            const float a = v[0] / (1.0f + expf(-v[0])) * v[1];
            if (f16_out_of_range(a)) atomicOr(p.status, QW_DEV_RANGE);
            __stcg(reinterpret_cast<unsigned short*>(p.act) + (size_t)t * p.I + row, __half_as_ushort(__float2half_rn(a)));
        });
        if (!(ok = gsync(ok))) break;

        // ---- down_proj + residual (Pasos 6, 7) ----------------------------------------
        stage_h(p.act, p.I);
        ok = consume_all(PH_D, l, false, [&](int row, int t, const float* v) {
            float* xp = p.x + (size_t)t * p.D + row;
            const float nv = __ldcg(xp) + v[0];
            __stcg(xp, nv);
            if (p.dbg_hidden) p.dbg_hidden[((size_t)l * T + t) * p.D + row] = nv;
        });
        if (!(ok = gsync(ok))) break;
    }

    // ---- final norm + tied LM head + greedy argmax (Paso 8) --------------------------------
    if (ok) {
        stage_norm(p.fnorm);
        unsigned long long best[MK_TMAX];
#pragma unroll
        for (int t = 0; t < MK_TMAX; ++t) best[t] = 0ull;
        const float rs_lane = lane < T ? rs_of(lane) : 0.f;  // this lane's token (lane = t below)
        ok = consume(PH_LM, 0, [&](int row, int t, const float* v) {
            const float y = v[0] * rs_lane;
            if (p.logits) __stcg(p.logits + (size_t)t * p.V + row, y);
#pragma unroll
            for (int q = 0; q < MK_TMAX; ++q)
                if (q == t) best[q] = u64_max(best[q], argmax_key(y, row));
        });
        if (!ok) s_fail = 1;
#pragma unroll
        for (int t = 0; t < MK_TMAX; ++t)
            if (t == lane) s_best[warp][t] = best[t];
        named_sync(1, MK_CONS_THREADS);
        ok = (s_fail == 0);
        if (ok && threadIdx.x < T) {
            unsigned long long b = 0ull;
            for (int w = 0; w < MK_CONS_WARPS; ++w) b = u64_max(b, s_best[w][threadIdx.x]);
            atomicMax(p.best + threadIdx.x, b);
        }
        __threadfence();
        named_sync(1, MK_CONS_THREADS);
        if (threadIdx.x == 0) s_last = ok && (atomicAdd(p.sync + 2, 1u) == G - 1);
        named_sync(1, MK_CONS_THREADS);
        if (s_last) {
            __threadfence();
            if (threadIdx.x < T) {
                const unsigned long long key = atomicExch(p.best + threadIdx.x, 0ull);
                p.next_ids[threadIdx.x] = (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
                p.kv.len[p.seq[threadIdx.x]] += 1;
            }
            if (threadIdx.x == 0) {
                atomicExch(p.sync + 2, 0u);
                atomicExch(p.sync, 0u);  // every CTA is past its last grid barrier
            }
        }
    }
    if (!ok) {
        // drain: wait (bounded, ignoring the abort word) for every ring stage the producer
        // issued and nobody consumed, so no bulk copy is in flight when the CTA exits
        const uint64_t t0 = globaltimer_ns();
        while (it < s_issued && globaltimer_ns() - t0 < kMkWaitNs) {
            const int st = it % MK_NST;
            if (mb_try(su32(full + st), (it / MK_NST) & 1u)) ++it;
        }
    }
}

namespace {
bool g_mk_attr = false;
}

int mk_smem_bytes() { return 1024 + MK_NST * MK_STAGE + MK_ACT + 2 * MK_NST * 8 + 64; }

// Largest T the persistent kernel handles for these dims (0 if none): fp32 activation
// rows must fit the 48 KB staging area and every matrix row must split into whole work
// items that fit a stage.
int mk_max_tokens(int D, int I, int QD) {
    int t = MK_TMAX;
    while (t > 0 && (t * D * 4 > MK_ACT || t * QD * 4 > MK_ACT || t * I * 4 > MK_ACT)) --t;
    for (int K : {D, I, QD})
        if (K % MK_SEG || K / MK_SEG > MK_ITEMS || MK_ITEMS % (K / MK_SEG)) return 0;
    if (MK_TEAMS * 1408 * 4 + 256 > MK_ACT) return 0;
    return t;
}

cudaError_t launch_decode_mk(const LaunchCtx& c, const MkParams& p, int grid) {
    const int smem = mk_smem_bytes();
    if (!g_mk_attr) {
        cudaError_t e = cudaFuncSetAttribute(k_decode_mk, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        g_mk_attr = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(MK_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (c.counter) ++*c.counter;
    return cudaLaunchKernelEx(&cfg, k_decode_mk, p);
}

int mk_grid_size() {
    int dev = 0, sms = 0, per = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (!g_mk_attr) {
        if (cudaFuncSetAttribute(k_decode_mk, cudaFuncAttributeMaxDynamicSharedMemorySize, mk_smem_bytes()) != cudaSuccess)
            return 0;
        g_mk_attr = true;
    }
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, k_decode_mk, MK_THREADS, mk_smem_bytes()) != cudaSuccess)
        return 0;
    return per >= 1 ? sms : 0;  // one CTA per SM
}
