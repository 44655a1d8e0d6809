// Grouped-query causal attention over the paged KV cache (Paso 5 of "Dentro de un LLM:
// Inferencia en Python puro para Qwen3-0.6B en MLX").
//
// k_attn_paged: split-KV flash-decode. One CTA per (query token, KV head, split of the
// key range); it serves both query heads of its KV head (head h reads KV head h / 2), so
// every K/V byte is loaded once for the two heads. Each of the 4 warps walks pages of 16
// keys with an online softmax in fp32 (exp2 domain); lanes split head_dim into 16-byte
// chunks and the two half-warps take alternate keys. Warps merge through shared memory;
// splits merge with log-sum-exp weights in the CTA that finishes last (an atomic ticket,
// no waiting). The query at position p sees keys 0..p of its sequence (the causal rule by
// position).
//
// Two modes. Prefill: the new tokens' K/V were appended by k_qknorm_rope_append and q is
// read as fp16. Decode (one new token per sequence, FUSED): the CTA itself applies the
// per-head QK-norm and rotate-half RoPE (Paso 5, Paso 4) to its two query heads and its KV
// head from the fp32 q|k|v projection row, keeps q in fp32, and the CTA whose split holds
// the new position appends the new K/V to its page slot before reading it back.
#include <algorithm>
#include <utility>

#include "qw_internal.h"
#include "tc_sm103.cuh"

namespace {

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ float dot8q(const float* q, const uint4 k) {
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

__device__ __forceinline__ float half_warp_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    return v;
}

}  // namespace

struct AttnP {
    const f16* q;       // [T][n_heads][128] (prefill mode)
    const float* qkv;   // [T][(n_heads + 2 n_kv) * 128] fp32 (decode mode)
    const bf16* q_norm; // [128]
    const bf16* k_norm; // [128]
    float eps;
    const float* rope_cos;  // [max_context][64]
    const float* rope_sin;
    int32_t* dbg_pos;
    int32_t* dbg_slot;
    int* status;
    int n_heads, n_kv;
    TokView tv;
    KVView kv;
    int layer;
    int chunk;          // keys per split (multiple of 16)
    int n_splits;       // grid.x; partial buffers have this many slots per (token, head)
    float* part_o;      // [T][n_heads][n_splits][128]
    float* part_ml;     // [T][n_heads][n_splits][2]
    int* counters;      // [T][n_kv]
    f16* out;           // [T][n_heads * 128]
    float scale_log2;   // head_dim^-0.5 * log2(e)
    // decode: sequence of each token (kernel parameter), so that the pages cached by earlier
    // steps can be prefetched into L2 before the dependency wait; prefetch = 0 turns it off
    int prefetch;
    int seqp[QW_MAX_BATCH];
};

constexpr int AW = 4;  // warps per CTA

__device__ __forceinline__ void prefetch_l2(const void* ptr, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}

template <bool FUSED>
__global__ void __launch_bounds__(AW * 32) k_attn_paged(const __grid_constant__ AttnP p) {
    pdl_launch();
    if (p.prefetch) {
        // the sequence length and page table were written before this step began (the step's
        // first kernel waits for everything earlier), so the first cached page of each warp
        // (the warps take pages round-robin) can be requested into L2 while the projection is
        // still running; only the first, so that a large batch does not overflow L2
        const int t = blockIdx.z, g = blockIdx.y, s = blockIdx.x;
        const int seq = p.seqp[t];
        const int len = p.kv.len[seq];
        const int k0 = s * p.chunk, k1 = min(k0 + p.chunk, len);
        const int* pt = p.kv.page_table + (size_t)seq * p.kv.max_pages_per_seq;
        const size_t lay = (size_t)p.layer * p.kv.layer_stride;
        const int pg = (k0 >> 4) + threadIdx.x;
        if (threadIdx.x < AW && pg < ((k1 + 15) >> 4)) {
            const int page = pt[pg];
            if (page >= 0 && page < p.kv.n_pages) {
                const size_t off = lay + ((size_t)page * p.n_kv + g) * 16 * 128;
                prefetch_l2(p.kv.k + off, 16 * 128 * 2);
                prefetch_l2(p.kv.v + off, 16 * 128 * 2);
            }
        }
    }
    pdl_wait();
    const int t = blockIdx.z, g = blockIdx.y, s = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int pos = p.tv.pos[t], seq = p.tv.seq[t];
    const int n_keys = pos + 1;
    const int n_act = (n_keys + p.chunk - 1) / p.chunk;
    if (s >= n_act) return;
    const int k0 = s * p.chunk, k1 = min(k0 + p.chunk, n_keys);
    const int half = lane >> 4, dl = (lane & 15) * 8;

    const int* pt = p.kv.page_table + (size_t)seq * p.kv.max_pages_per_seq;
    const bool writer = FUSED && (s == n_act - 1);  // this split holds the new position
    __shared__ float sq[2][128];
    if (FUSED) {
        // warp 0, 1: query heads 2g, 2g+1; warp 2: KV head g's key; warp 3: its value
        const int NH = p.n_heads + 2 * p.n_kv;
        const int hh = warp < 2 ? 2 * g + warp : (warp == 2 ? p.n_heads + g : p.n_heads + p.n_kv + g);
        const float4 xv = *reinterpret_cast<const float4*>(p.qkv + ((size_t)t * NH + hh) * 128 + lane * 4);
        float y[4] = {xv.x, xv.y, xv.z, xv.w};
        if (warp < 3) {
            const bf16* nw = warp < 2 ? p.q_norm : p.k_norm;
            const float ss = warp_sum(y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3]);
            const float r = rsqrtf(ss * (1.0f / 128.0f) + p.eps);
            const uint2 wb = *reinterpret_cast<const uint2*>(nw + lane * 4);
            y[0] *= r * bf_lo(wb.x);
            y[1] *= r * bf_hi(wb.x);
            y[2] *= r * bf_lo(wb.y);
            y[3] *= r * bf_hi(wb.y);
            const int i0 = (lane & 15) * 4;
            const float4 cs = *reinterpret_cast<const float4*>(p.rope_cos + (size_t)pos * 64 + i0);
            const float4 sn = *reinterpret_cast<const float4*>(p.rope_sin + (size_t)pos * 64 + i0);
            const float c[4] = {cs.x, cs.y, cs.z, cs.w}, sv[4] = {sn.x, sn.y, sn.z, sn.w};
            float o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float pj = __shfl_xor_sync(0xffffffffu, y[j], 16);
                o[j] = (lane < 16) ? (y[j] * c[j] - pj * sv[j]) : (pj * sv[j] + y[j] * c[j]);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) y[j] = o[j];
        }
        if (warp < 2) {
#pragma unroll
            for (int j = 0; j < 4; ++j) sq[warp][lane * 4 + j] = y[j];
        } else if (writer) {
            const int pi = pos >> 4;
            const int page = (pi < p.kv.max_pages_per_seq) ? pt[pi] : -1;
            if (page < 0 || page >= p.kv.n_pages) {
                if (lane == 0) atomicOr(p.status, QW_DEV_BAD_POS);
            } else {
                f16* pool = (warp == 2 ? p.kv.k : p.kv.v) + (size_t)p.layer * p.kv.layer_stride;
                if (f16_out_of_range(y[0]) || f16_out_of_range(y[1]) || f16_out_of_range(y[2]) ||
                    f16_out_of_range(y[3]))
                    atomicOr(p.status, QW_DEV_RANGE);
                uint2 packed;
                packed.x = pack_h2(y[0], y[1]);
                packed.y = pack_h2(y[2], y[3]);
                *reinterpret_cast<uint2*>(pool + (((size_t)page * p.n_kv + g) * 16 + (pos & 15)) * 128 + lane * 4) =
                    packed;
                if (p.dbg_pos && warp == 2 && g == 0 && lane == 0) {
                    p.dbg_pos[t] = pos;
                    p.dbg_slot[t] = page * 16 + (pos & 15);
                }
            }
        }
        __syncthreads();
    }
    float q0[8], q1[8];
    if (FUSED) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            q0[i] = sq[0][dl + i] * p.scale_log2;
            q1[i] = sq[1][dl + i] * p.scale_log2;
        }
    } else {
        const f16* qp = p.q + ((size_t)t * p.n_heads + 2 * g) * 128 + dl;
        const uint4 a = *reinterpret_cast<const uint4*>(qp);
        const uint4 b = *reinterpret_cast<const uint4*>(qp + 128);
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            q0[2 * i] = h_lo(aw[i]) * p.scale_log2;
            q0[2 * i + 1] = h_hi(aw[i]) * p.scale_log2;
            q1[2 * i] = h_lo(bw[i]) * p.scale_log2;
            q1[2 * i + 1] = h_hi(bw[i]) * p.scale_log2;
        }
    }
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o0[8], o1[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o0[i] = o1[i] = 0.f;

    const f16* Kl = p.kv.k + (size_t)p.layer * p.kv.layer_stride;
    const f16* Vl = p.kv.v + (size_t)p.layer * p.kv.layer_stride;
    const int p0 = k0 >> 4, p1 = (k1 + 15) >> 4;

    for (int pg = p0 + warp; pg < p1; pg += AW) {
        const int page = pt[pg];
        if (page < 0 || page >= p.kv.n_pages) continue;  // reported by the append kernel
        const int nvalid = min(16, k1 - pg * 16);
        const size_t off = ((size_t)page * p.n_kv + g) * 16 * 128 + dl;
        uint4 kr[8], vr[8];
        if (writer && pg == p1 - 1) {
            // the page this CTA just wrote: coherent loads (not the read-only path)
#pragma unroll
            for (int i = 0; i < 8; ++i) kr[i] = *reinterpret_cast<const uint4*>(Kl + off + (size_t)(2 * i + half) * 128);
#pragma unroll
            for (int i = 0; i < 8; ++i) vr[i] = *reinterpret_cast<const uint4*>(Vl + off + (size_t)(2 * i + half) * 128);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) kr[i] = ldg_nc(Kl + off + (size_t)(2 * i + half) * 128);
#pragma unroll
            for (int i = 0; i < 8; ++i) vr[i] = ldg_nc(Vl + off + (size_t)(2 * i + half) * 128);
        }
        // slots past the last valid key hold whatever the pool held before: give them zero
        // values as well as zero weight (0 * NaN would poison the sum)
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (2 * i + half >= nvalid) vr[i] = make_uint4(0u, 0u, 0u, 0u);
        float s0[8], s1[8];
        float pm0 = -INFINITY, pm1 = -INFINITY;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float d0 = half_warp_sum(dot8q(q0, kr[i]));
            const float d1 = half_warp_sum(dot8q(q1, kr[i]));
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
    // the two half-warps saw alternate keys with the same running max
    l0 += __shfl_xor_sync(0xffffffffu, l0, 16);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 16);
#pragma unroll
    for (int d = 0; d < 8; ++d) {
        o0[d] += __shfl_xor_sync(0xffffffffu, o0[d], 16);
        o1[d] += __shfl_xor_sync(0xffffffffu, o1[d], 16);
    }

    __shared__ float sm_o[AW][2][128];
    __shared__ float sm_m[AW][2], sm_l[AW][2];
    __shared__ int sm_last;
    if (lane < 16) {
#pragma unroll
        for (int d = 0; d < 8; ++d) {
            sm_o[warp][0][dl + d] = o0[d];
            sm_o[warp][1][dl + d] = o1[d];
        }
    }
    if (lane == 0) {
        sm_m[warp][0] = m0;
        sm_m[warp][1] = m1;
        sm_l[warp][0] = l0;
        sm_l[warp][1] = l1;
    }
    __syncthreads();

    // 128 threads: thread -> (head hh, dims 2*(tid%64), +1)
    const int hh = threadIdx.x >> 6, d2 = (threadIdx.x & 63) * 2;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < AW; ++w) M = fmaxf(M, sm_m[w][hh]);
    float L = 0.f, O0 = 0.f, O1 = 0.f;
#pragma unroll
    for (int w = 0; w < AW; ++w) {
        const float f = exp2f(sm_m[w][hh] - M);
        L += sm_l[w][hh] * f;
        O0 += sm_o[w][hh][d2] * f;
        O1 += sm_o[w][hh][d2 + 1] * f;
    }
    const int head = 2 * g + hh;
    f16* outp = p.out + ((size_t)t * p.n_heads + head) * 128 + d2;
    if (n_act == 1) {
        *reinterpret_cast<uint32_t*>(outp) = pack_h2(O0 / L, O1 / L);
        return;
    }
    const size_t slot = ((size_t)t * p.n_heads + head) * p.n_splits + s;
    *reinterpret_cast<float2*>(p.part_o + slot * 128 + d2) = make_float2(O0, O1);
    if ((threadIdx.x & 63) == 0) *reinterpret_cast<float2*>(p.part_ml + slot * 2) = make_float2(M, L);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const int ticket = atomicAdd(p.counters + (size_t)t * p.n_kv + g, 1);
        sm_last = (ticket == n_act - 1);
    }
    __syncthreads();
    if (!sm_last) return;
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
    *reinterpret_cast<uint32_t*>(outp) = pack_h2(A0 / LL, A1 / LL);
    if (threadIdx.x == 0) p.counters[(size_t)t * p.n_kv + g] = 0;
}

cudaError_t launch_attn_paged(const LaunchCtx& c, int T, int layer, const f16* q, int n_heads,
                              int n_kv, TokView tv, KVView kv, int chunk, int n_splits,
                              float* part_o, float* part_ml, int* counters, f16* out,
                              const AttnFuse* fuse, const int* decode_seqs) {
    AttnP p = {};
    if (decode_seqs) {
        p.prefetch = 1;
        for (int t = 0; t < T; ++t) p.seqp[t] = decode_seqs[t];
    }
    p.q = q;
    p.n_heads = n_heads;
    p.n_kv = n_kv;
    p.tv = tv;
    p.kv = kv;
    p.layer = layer;
    p.chunk = chunk;
    p.n_splits = n_splits;
    p.part_o = part_o;
    p.part_ml = part_ml;
    p.counters = counters;
    p.out = out;
    p.scale_log2 = 0.08838834764831845f * 1.4426950408889634f;  // 128^-0.5 * log2(e)
    if (fuse) {
        p.qkv = fuse->qkv;
        p.q_norm = fuse->q_norm;
        p.k_norm = fuse->k_norm;
        p.eps = fuse->eps;
        p.rope_cos = fuse->rope_cos;
        p.rope_sin = fuse->rope_sin;
        p.dbg_pos = fuse->dbg_pos;
        p.dbg_slot = fuse->dbg_slot;
        p.status = fuse->status;
        return launch_k(c, k_attn_paged<true>, dim3(n_splits, n_kv, T), dim3(AW * 32), 0, p);
    }
    return launch_k(c, k_attn_paged<false>, dim3(n_splits, n_kv, T), dim3(AW * 32), 0, p);
}

// =======================================================================================
// k_attn_oproj: decode attention of ONE token over a short cache fused with o_proj (Pasos 5
// and 7), for the latency-bound batch-1 decode step. o_proj is split by KV head: with heads
// 2g, 2g+1 reading KV head g, the 256 attention outputs of g are exactly inputs
// [256 g, 256 g + 256) of o_proj, so x += Wo o becomes x += sum_g Wo[:, 256 g ..] o_g. CTA
// (rb, g) computes the attention of KV head g -- QK-norm and RoPE of its two query heads and
// of the new key, online softmax over the cached pages plus the new key (taken from
// registers, rounded to fp16 as the cache stores it) -- and the partial product of o_proj rows
// [32 rb, 32 rb + 32) over that head's inputs into part[g][row]. The 32 CTAs of a head repeat
// its attention (a few cached pages) instead of waiting for each other; the CTAs with rb == 0
// append the new K/V. The partials are added to x, in order of g, by the next kernels
// (gate/up reads x + sum_g part[g] for its RMSNorm, down_proj adds them to the residual it
// updates). Nothing of the cached pages or of o_proj depends on the step, so before the
// dependency wait each CTA loads its o_proj weights into registers and bulk-copies the head's
// cached K/V pages (at most AO_MAXPG) into shared memory.
// =======================================================================================
namespace {

constexpr int AO_ROWS = 32;    // o_proj rows per CTA (8 per warp)
constexpr int AO_MAXPG = 12;   // cached pages held in shared memory (192 keys)
constexpr int AO_PAGE = 16 * 128 * 2;  // K (or V) of one 16-key page of one head (4 KB)
constexpr unsigned long long AO_WAIT_NS = 2000000000ull;

struct AttnOP {
    const float* qkv;  // [(n_heads + 2 n_kv) * 128] fp32
    const bf16* q_norm;
    const bf16* k_norm;
    float eps;
    const float* rope_cos;
    const float* rope_sin;
    int32_t* dbg_pos;
    int32_t* dbg_slot;
    int* status;
    f16* dbg_attn;  // optional [n_heads * 128]
    int n_heads, n_kv, D, QD;
    int seq;        // the token's sequence (its cached length and pages are read before the wait)
    TokView tv;
    KVView kv;
    int layer;
    const bf16* Wo;  // [D][QD] of this layer
    float* part;     // [n_kv][D]
    float scale_log2;
};

__device__ __forceinline__ float dot8_bf(const uint4 w, const float4 a0, const float4 a1) {
    float acc = bf_lo(w.x) * a0.x;
    acc = fmaf(bf_hi(w.x), a0.y, acc);
    acc = fmaf(bf_lo(w.y), a0.z, acc);
    acc = fmaf(bf_hi(w.y), a0.w, acc);
    acc = fmaf(bf_lo(w.z), a1.x, acc);
    acc = fmaf(bf_hi(w.z), a1.y, acc);
    acc = fmaf(bf_lo(w.w), a1.z, acc);
    acc = fmaf(bf_hi(w.w), a1.w, acc);
    return acc;
}

}  // namespace

__global__ void __launch_bounds__(128) k_attn_oproj(const __grid_constant__ AttnOP p) {
    extern __shared__ __align__(128) uint8_t ao_pages[];  // [page][K 4 KB | V 4 KB]
    __shared__ __align__(8) uint64_t ao_bar;
    __shared__ int ao_np, ao_bad;
    pdl_launch();
    const int rb = blockIdx.x, g = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const f16* Kl = p.kv.k + (size_t)p.layer * p.kv.layer_stride;
    const f16* Vl = p.kv.v + (size_t)p.layer * p.kv.layer_stride;
    const int* pt = p.kv.page_table + (size_t)p.seq * p.kv.max_pages_per_seq;
    // before the wait: the cached pages of head g (the length and page table were written
    // before this step began) and this CTA's o_proj weights
    if (threadIdx.x == 0) {
        const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&ao_bar);
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        const int cached = p.kv.len[p.seq];
        const int np = min((cached + 15) >> 4, AO_MAXPG);
        int bad = 0;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(np * 2 * AO_PAGE) : "memory");
        for (int i = 0; i < np; ++i) {
            int page = pt[i];
            if (page < 0 || page >= p.kv.n_pages) {
                bad = 1;  // reported by the append; any valid block keeps the copy in bounds
                page = 0;
            }
            const size_t off = ((size_t)page * p.n_kv + g) * 16 * 128;
            const uint32_t dst = (uint32_t)__cvta_generic_to_shared(ao_pages + (size_t)i * 2 * AO_PAGE);
            asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                         "l"(Kl + off), "r"(AO_PAGE), "r"(bar)
                         : "memory");
            asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst + AO_PAGE),
                         "l"(Vl + off), "r"(AO_PAGE), "r"(bar)
                         : "memory");
        }
        ao_np = np;
        ao_bad = bad;
    }
    uint4 wo[8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
        wo[r] = ldg_nc(p.Wo + (size_t)(rb * AO_ROWS + warp * 8 + r) * p.QD + 256 * g + lane * 8);
    pdl_wait();

    __shared__ float sq[2][128];            // rotated q of heads 2g, 2g+1
    __shared__ float skv[2][128];           // the new k (rotated) and v, as fp16 values
    __shared__ float so[4][2][128];         // per-warp partial outputs
    __shared__ float smm[4][2], sll[4][2];  // per-warp running max / sum
    __shared__ __align__(16) float ob[256]; // attention output of head pair g, fp16 values
    const int NH = p.n_heads + 2 * p.n_kv;
    const int half = lane >> 4, dl = (lane & 15) * 8;
    const int pos = p.tv.pos[0];
    // 1. QK-norm + RoPE of the query heads (warps 0, 1) and the new key (warp 2); v (warp 3)
    {
        const int hh = warp < 2 ? 2 * g + warp : (warp == 2 ? p.n_heads + g : p.n_heads + p.n_kv + g);
        const float4 xv = *reinterpret_cast<const float4*>(p.qkv + (size_t)hh * 128 + lane * 4);
        float y[4] = {xv.x, xv.y, xv.z, xv.w};
        if (warp < 3) {
            const bf16* nw = warp < 2 ? p.q_norm : p.k_norm;
            const float ss = warp_sum(y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3]);
            const float r = rsqrtf(ss * (1.0f / 128.0f) + p.eps);
            const uint2 wb = *reinterpret_cast<const uint2*>(nw + lane * 4);
            y[0] *= r * bf_lo(wb.x);
            y[1] *= r * bf_hi(wb.x);
            y[2] *= r * bf_lo(wb.y);
            y[3] *= r * bf_hi(wb.y);
            const int i0 = (lane & 15) * 4;
            const float4 cs = *reinterpret_cast<const float4*>(p.rope_cos + (size_t)pos * 64 + i0);
            const float4 sn = *reinterpret_cast<const float4*>(p.rope_sin + (size_t)pos * 64 + i0);
            const float c[4] = {cs.x, cs.y, cs.z, cs.w}, sv[4] = {sn.x, sn.y, sn.z, sn.w};
            float o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float pj = __shfl_xor_sync(0xffffffffu, y[j], 16);
                o[j] = (lane < 16) ? (y[j] * c[j] - pj * sv[j]) : (pj * sv[j] + y[j] * c[j]);
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
            if (rb == 0) {  // one CTA per KV head appends
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
    // the cached pages have landed (bounded wait)
    {
        const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&ao_bar);
        const uint64_t t0 = globaltimer_ns();
        uint32_t done = 0;
        while (true) {
            asm volatile(
                "{\n\t.reg .pred q;\n\t"
                "mbarrier.try_wait.parity.shared::cta.b64 q, [%1], 0;\n\t"
                "selp.u32 %0, 1, 0, q;\n\t}"
                : "=r"(done)
                : "r"(bar)
                : "memory");
            if (done) break;
            if (globaltimer_ns() - t0 > AO_WAIT_NS) {
                if (threadIdx.x == 0) atomicOr(p.status, QW_DEV_TIMEOUT);
                break;
            }
        }
    }
    __syncthreads();
    // 2. online softmax over the cached keys [0, pos) (pages round-robin over the warps; the
    //    page of the new position only below it) and, on warp 0, the new key
    float q0[8], q1[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        q0[i] = sq[0][dl + i] * p.scale_log2;
        q1[i] = sq[1][dl + i] * p.scale_log2;
    }
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, o0[8], o1[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o0[i] = o1[i] = 0.f;
    const int np = ao_np;
    for (int pg = warp; pg < np && !ao_bad; pg += 4) {
        const int nvalid = min(16, pos - pg * 16);
        const uint8_t* kp = ao_pages + (size_t)pg * 2 * AO_PAGE;
        uint4 kr[8], vr[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            kr[i] = *reinterpret_cast<const uint4*>(kp + ((2 * i + half) * 128 + dl) * 2);
            vr[i] = *reinterpret_cast<const uint4*>(kp + AO_PAGE + ((2 * i + half) * 128 + dl) * 2);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (2 * i + half >= nvalid) vr[i] = make_uint4(0u, 0u, 0u, 0u);
        float s0[8], s1[8], pm0 = -INFINITY, pm1 = -INFINITY;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float d0 = half_warp_sum(dot8q(q0, kr[i]));
            const float d1 = half_warp_sum(dot8q(q1, kr[i]));
            const bool valid = (2 * i + half) < nvalid;
            s0[i] = valid ? d0 : -INFINITY;
            s1[i] = valid ? d1 : -INFINITY;
            pm0 = fmaxf(pm0, s0[i]);
            pm1 = fmaxf(pm1, s1[i]);
        }
        pm0 = fmaxf(pm0, __shfl_xor_sync(0xffffffffu, pm0, 16));
        pm1 = fmaxf(pm1, __shfl_xor_sync(0xffffffffu, pm1, 16));
        const float n0 = fmaxf(m0, pm0), n1 = fmaxf(m1, pm1);
        if (n0 == -INFINITY) continue;
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
    if (warp == 0) {
        // the new key: both half-warps move the max, half 0 adds its weight
        float d0 = 0.f, d1 = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            d0 = fmaf(q0[i], skv[0][dl + i], d0);
            d1 = fmaf(q1[i], skv[0][dl + i], d1);
        }
        d0 = half_warp_sum(d0);
        d1 = half_warp_sum(d1);
        const float n0 = fmaxf(m0, d0), n1 = fmaxf(m1, d1);
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
        if (half == 0) {
            const float e0 = exp2f(d0 - m0), e1 = exp2f(d1 - m1);
            l0 += e0;
            l1 += e1;
#pragma unroll
            for (int d = 0; d < 8; ++d) {
                o0[d] = fmaf(e0, skv[1][dl + d], o0[d]);
                o1[d] = fmaf(e1, skv[1][dl + d], o1[d]);
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
            so[warp][0][dl + d] = o0[d];
            so[warp][1][dl + d] = o1[d];
        }
    }
    if (lane == 0) {
        smm[warp][0] = m0;
        smm[warp][1] = m1;
        sll[warp][0] = l0;
        sll[warp][1] = l1;
    }
    __syncthreads();
    {
        // 128 threads: thread -> (head hh, dims 2*(tid%64), +1); warps without keys add nothing
        const int hh = threadIdx.x >> 6, d2 = (threadIdx.x & 63) * 2;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, smm[w][hh]);
        float L = 0.f, O0 = 0.f, O1 = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float f = smm[w][hh] == -INFINITY ? 0.f : exp2f(smm[w][hh] - M);
            L += sll[w][hh] * f;
            O0 += so[w][hh][d2] * f;
            O1 += so[w][hh][d2 + 1] * f;
        }
        const uint32_t hv = pack_h2(O0 / L, O1 / L);  // the attention output as the unfused path stores it
        ob[hh * 128 + d2] = h_lo(hv);
        ob[hh * 128 + d2 + 1] = h_hi(hv);
        if (p.dbg_attn && rb == 0)
            *reinterpret_cast<uint32_t*>(p.dbg_attn + (size_t)(2 * g + hh) * 128 + d2) = hv;
    }
    __syncthreads();
    // 3. o_proj partial of this CTA's rows over KV head g's inputs
    const float4 a0 = *reinterpret_cast<const float4*>(&ob[lane * 8]);
    const float4 a1 = *reinterpret_cast<const float4*>(&ob[lane * 8 + 4]);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const float acc = warp_sum(dot8_bf(wo[r], a0, a1));
        if (lane == 0) p.part[(size_t)g * p.D + rb * AO_ROWS + warp * 8 + r] = acc;
    }
}

int attn_oproj_max_keys() { return AO_MAXPG * 16; }

cudaError_t launch_attn_oproj(const LaunchCtx& c, int seq, int layer, const AttnFuse& fz, int n_heads, int n_kv,
                              TokView tv, KVView kv, const bf16* Wo, int D, float* part, f16* dbg_attn) {
    if (D % AO_ROWS) return cudaErrorInvalidValue;
    static bool attr_set = false;
    const int smem = AO_MAXPG * 2 * AO_PAGE;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_attn_oproj, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    AttnOP p = {};
    p.qkv = fz.qkv;
    p.q_norm = fz.q_norm;
    p.k_norm = fz.k_norm;
    p.eps = fz.eps;
    p.rope_cos = fz.rope_cos;
    p.rope_sin = fz.rope_sin;
    p.dbg_pos = fz.dbg_pos;
    p.dbg_slot = fz.dbg_slot;
    p.status = fz.status;
    p.dbg_attn = dbg_attn;
    p.n_heads = n_heads;
    p.n_kv = n_kv;
    p.D = D;
    p.QD = n_heads * 128;
    p.seq = seq;
    p.tv = tv;
    p.kv = kv;
    p.layer = layer;
    p.Wo = Wo;
    p.part = part;
    p.scale_log2 = 0.08838834764831845f * 1.4426950408889634f;  // 128^-0.5 * log2(e)
    return launch_k(c, k_attn_oproj, dim3(D / AO_ROWS, n_kv), dim3(128), (size_t)smem, p);
}

// =======================================================================================
// Warp-level helpers of the mma.sync paths (decode attention) and of the prefill kernel's
// Q staging: cp.async copies, ldmatrix, m16n8k16 MMA.
// =======================================================================================
namespace {

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

}  // namespace

// 2^x with the hardware approximation (PTX ex2.approx.ftz; 2^-inf = +0), for the softmax
// weights of the prefill attention
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// =======================================================================================
// k_attn_decode: decode attention over long or many caches (Paso 5), one new token per
// sequence, q already normalised and rotated (fp16) and its K/V already in the cache.
//
// The work items (token t, KV head g, page i) are laid out token-major, then head, then page,
// and split into equal contiguous ranges over a fixed grid (2 CTAs per SM), so ragged cache
// lengths cost no load imbalance and no wave tail. A CTA walks its range as segments (the
// pages of one (t, g) pair inside the range). A producer warp streams each page's K and V
// blocks with TMA tensor copies (the pools seen as [rows, 128] fp16, boxes of 16 rows x 64
// dims with the 128-byte swizzle) into a 12-stage shared-memory ring; four consumer warps take
// the pages of a segment round-robin. Per page a warp computes S = Q K^T and O += P V with
// mma.sync m16n8k16 (fp16 operands, fp32 accumulation; the two query heads 2g, 2g+1 are rows
// 0 and 1 of a 16-row tile), keeping the online softmax in fp32 in the exp2 domain. A segment
// that covers its whole pair writes the output; otherwise the partial (m, l, o) goes to its
// slot and the CTA that finishes the pair last (atomic ticket, no waiting) merges the slots
// in order. Cache lengths and page tables were written before the step began, so the ring is
// filled before the dependency wait, except a pair's newest page, which the kernel that
// precedes this one writes.
// =======================================================================================
namespace {

constexpr int AD_CW = 4;                      // consumer warps
constexpr int AD_THREADS = (AD_CW + 1) * 32;  // + producer warp
constexpr int AD_NST = 12;                    // ring stages
// Within a segment consumer warp w takes items k = k_base + w, + CW, ...; it waits for a
// stage by phase parity, which is sound only if the previous use of the same stage (item
// k - NST) was its own (or belongs to an earlier segment, closed by the merge barrier).
static_assert(AD_NST % AD_CW == 0, "ring depth must be a multiple of the consumer warps");
constexpr int AD_BOX = 16 * 128;              // bytes of one 16-row x 64-dim box
constexpr int AD_STAGE = 4 * AD_BOX;          // K dims 0-63, K 64-127, V 0-63, V 64-127
constexpr unsigned long long AD_WAIT_NS = 2000000000ull;

__device__ __forceinline__ uint32_t ad_smem(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ bool ad_try_wait(uint32_t bar, uint32_t parity) {
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

// bounded wait; false after ~2 s or when another role gave up
__device__ __forceinline__ bool ad_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (ad_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    uint32_t n = 0;
    while (true) {
        if (ad_try_wait(bar, parity)) return true;
        if ((++n & 255u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > AD_WAIT_NS) return false;
        }
    }
}

// the CTA whose item range [c N / G, (c + 1) N / G) holds item j
__device__ __forceinline__ int ad_cta_of(long long j, long long N, int G) {
    return (int)(((j + 1) * G - 1) / N);
}

// byte offset of 16-byte chunk `ch` (0..7) of row r inside a 128-byte-swizzled box
__device__ __forceinline__ uint32_t ad_swz(int r, int ch) { return (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4)); }

__device__ __forceinline__ void ad_tma_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

}  // namespace

struct AttnDP {
    CUtensorMap tmK;     // K pool [n_layers * n_pages * n_kv * 16, 128] fp16
    CUtensorMap tmV;
    const f16* q;        // [T][n_heads][128]
    f16* out;            // [T][n_heads][128]
    KVView kv;
    int layer, n_heads, n_kv, T;
    float* part_o;       // [T][n_heads][max_slots][128]
    float* part_ml;      // [T][n_heads][max_slots][2]
    int* counters;       // [T][n_kv], zero between launches
    int max_slots;
    int* status;
    float scale_log2;
    int seqp[QW_MAX_BATCH];  // sequence of each token
};

// shared-memory layout of k_attn_decode (byte offsets from a 1024-aligned base)
constexpr int AD_OFF_FULL = AD_NST * AD_STAGE;                 // ring first
constexpr int AD_OFF_EMPTY = AD_OFF_FULL + AD_NST * 8;
constexpr int AD_OFF_FLAGS = AD_OFF_EMPTY + AD_NST * 8;
constexpr int AD_OFF_PREF = AD_OFF_FLAGS + 16;                 // [T + 1] page prefix
constexpr int AD_OFF_NKEY = AD_OFF_PREF + ((QW_MAX_BATCH + 1) * 4 + 15) / 16 * 16;  // [T] keys
constexpr int AD_OFF_SMO = AD_OFF_NKEY + QW_MAX_BATCH * 4;     // [CW][2][128]
constexpr int AD_OFF_SMM = AD_OFF_SMO + AD_CW * 2 * 128 * 4;   // [CW][2]
constexpr int AD_OFF_SML = AD_OFF_SMM + AD_CW * 2 * 4;         // [CW][2]
constexpr int AD_SMEM = 1024 + AD_OFF_SML + AD_CW * 2 * 4;     // + alignment slack
static_assert(AD_OFF_FULL % 8 == 0 && AD_OFF_PREF % 16 == 0, "alignment");

__global__ void __launch_bounds__(AD_THREADS) k_attn_decode(const __grid_constant__ AttnDP p) {
    extern __shared__ uint8_t ad_raw_[];
    uint8_t* ad_raw = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ad_raw_) + 1023) & ~(uintptr_t)1023);
    uint8_t* ring = ad_raw;
    uint64_t* full = reinterpret_cast<uint64_t*>(ad_raw + AD_OFF_FULL);
    uint64_t* empty = reinterpret_cast<uint64_t*>(ad_raw + AD_OFF_EMPTY);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(ad_raw + AD_OFF_FLAGS);
    volatile int* last_flag = abort_flag + 1;
    int* pref = reinterpret_cast<int*>(ad_raw + AD_OFF_PREF);
    int* nkey = reinterpret_cast<int*>(ad_raw + AD_OFF_NKEY);
    float* sm_o = reinterpret_cast<float*>(ad_raw + AD_OFF_SMO);
    float* sm_m = reinterpret_cast<float*>(ad_raw + AD_OFF_SMM);
    float* sm_l = reinterpret_cast<float*>(ad_raw + AD_OFF_SML);

    pdl_launch();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = p.T, G = gridDim.x, c = blockIdx.x;
    // ---- work layout (cache lengths are stable during the step: before the wait) ----------
    for (int t = tid; t < T; t += AD_THREADS) nkey[t] = p.kv.len[p.seqp[t]] + 1;
    if (tid == 0) {
        for (int s = 0; s < AD_NST; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(ad_smem(full + s)) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(ad_smem(empty + s)) : "memory");
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == AD_CW && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&p.tmK) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&p.tmV) : "memory");
    }
    __syncthreads();
    if (warp == 0) {  // exclusive prefix of pages per token
        int run = 0;
        for (int t0 = 0; t0 < T; t0 += 32) {
            const int t = t0 + lane;
            const int v = t < T ? (nkey[t] + 15) >> 4 : 0;
            int x = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (t < T) pref[t] = run + x - v;
            run += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) pref[T] = run;
    }
    __syncthreads();
    const long long N = (long long)p.n_kv * pref[T];
    const long long i_begin = (long long)c * N / G, i_end = (long long)(c + 1) * N / G;

    // segment iterator: item j -> token t (largest with n_kv * pref[t] <= j), head, page
    auto segment = [&](long long j, int& t, int& g, int& i0, int& n) {
        int lo = 0, hi = T - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((long long)p.n_kv * pref[mid] <= j) lo = mid; else hi = mid - 1;
        }
        t = lo;
        const int np = pref[t + 1] - pref[t];
        const long long rel = j - (long long)p.n_kv * pref[t];
        g = (int)(rel / np);
        i0 = (int)(rel % np);
        const long long seg_end = min(i_end, (long long)p.n_kv * pref[t] + (long long)(g + 1) * np);
        n = (int)(seg_end - j);
    };

    if (warp == AD_CW) {
        // ---------------- producer (the whole warp; lane 0 issues) ----------------
        // page ids are fetched 32 at a time, one per lane, so the issue loop does not wait
        // on a page-table load per page
        bool waited = false;
        int k = 0;
        const long long layer_rows = (long long)p.layer * p.kv.n_pages;
        for (long long j = i_begin; j < i_end && !*abort_flag;) {
            int t, g, i0, n;
            segment(j, t, g, i0, n);
            const int* pt = p.kv.page_table + (size_t)p.seqp[t] * p.kv.max_pages_per_seq;
            const int newest = ((nkey[t] + 15) >> 4) - 1;
            bool stop = false;
            for (int c0 = 0; c0 < n && !stop; c0 += 32) {
                const int il = i0 + c0 + lane;
                int pid = (c0 + lane < n && il < p.kv.max_pages_per_seq) ? pt[il] : -1;
                if (c0 + lane < n && (pid < 0 || pid >= p.kv.n_pages)) {
                    atomicOr(p.status, QW_DEV_BAD_POS);
                    pid = 0;  // any valid block; the result is flagged
                }
                const int cn = min(32, n - c0);
                for (int jj = 0; jj < cn; ++jj, ++k) {
                    const int page = __shfl_sync(0xffffffffu, pid, jj);
                    const int i = i0 + c0 + jj;
                    if (!waited && i == newest) {  // written by the preceding kernel
                        pdl_wait();
                        waited = true;
                    }
                    const int s = k % AD_NST;
                    int ok = 1;
                    if (lane == 0 && k >= AD_NST && !ad_wait(ad_smem(empty + s), ((k / AD_NST) & 1) ^ 1, abort_flag)) {
                        *abort_flag = 1;
                        ok = 0;
                    }
                    if (!__shfl_sync(0xffffffffu, ok, 0)) {
                        stop = true;
                        break;
                    }
                    if (lane == 0) {
                        const int row = (int)(((layer_rows + page) * p.n_kv + g) * 16);
                        const uint32_t dst = ad_smem(ring + s * AD_STAGE), bar = ad_smem(full + s);
                        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(AD_STAGE)
                                     : "memory");
                        ad_tma_2d(dst, &p.tmK, bar, 0, row);
                        ad_tma_2d(dst + AD_BOX, &p.tmK, bar, 64, row);
                        ad_tma_2d(dst + 2 * AD_BOX, &p.tmV, bar, 0, row);
                        ad_tma_2d(dst + 3 * AD_BOX, &p.tmV, bar, 64, row);
                    }
                }
            }
            j += n;
        }
        if (!waited) pdl_wait();
        // before the CTA can retire, every copy issued must have landed (at once on the
        // normal path; bounded when the consumers gave up)
        if (lane == 0) {
            for (int kk = max(0, k - AD_NST); kk < k; ++kk) {
                const uint32_t bar = ad_smem(full + kk % AD_NST), par = (kk / AD_NST) & 1;
                const uint64_t t0 = globaltimer_ns();
                while (!ad_try_wait(bar, par) && globaltimer_ns() - t0 < AD_WAIT_NS) {
                }
            }
        }
        return;  // the producer takes no part in the consumers' named barriers
    }

    // ---------------- consumers ----------------
    pdl_wait();  // q is written by the preceding kernel
    const int gq = lane >> 2, tq = lane & 3;  // mma fragment row group / column pair
    int k_base = 0;
    for (long long j = i_begin; j < i_end;) {
        int t, g, i0, n;
        segment(j, t, g, i0, n);
        // Q as the A operand: rows 0 and 1 = heads 2g, 2g+1 (lanes 0-7); rows 2-15 are zero
        uint32_t qa[8][2];  // per k-step: (row gq, dims 16ks + 2tq..) and (row gq, dims +8)
        {
            const bool live = gq < 2;
            const f16* qp = p.q + ((size_t)t * p.n_heads + 2 * g + (live ? gq : 0)) * 128 + 2 * tq;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                qa[ks][0] = live ? *reinterpret_cast<const uint32_t*>(qp + 16 * ks) : 0u;
                qa[ks][1] = live ? *reinterpret_cast<const uint32_t*>(qp + 16 * ks + 8) : 0u;
            }
        }
        float m_r = -INFINITY, l_r = 0.f;  // this lane's row (head gq for lanes 0-7)
        float o[16][4];
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
        const int nk = nkey[t];
        for (int jj = warp; jj < n; jj += AD_CW) {
            const int k = k_base + jj, s = k % AD_NST;
            if (*abort_flag) continue;
            if (!ad_wait(ad_smem(full + s), (k / AD_NST) & 1, abort_flag)) {
                *abort_flag = 1;
                atomicOr(p.status, QW_DEV_TIMEOUT);
                continue;
            }
            uint8_t* st = ring + s * AD_STAGE;
            const uint32_t sa = ad_smem(st);
            const int nvalid = min(16, nk - (i0 + jj) * 16);
            if (nvalid < 16) {
                // slots past the last key hold stale pool data (possibly not finite): zero
                // their V rows so that 0-weight keys add exactly nothing
                for (int e = lane; e < (16 - nvalid) * 16; e += 32) {
                    const int r = nvalid + (e >> 4), box = 2 + ((e >> 3) & 1), ch = e & 7;
                    *reinterpret_cast<uint4*>(st + box * AD_BOX + ad_swz(r, ch)) = make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
            }
            // ---- S = Q K^T: 16 rows x 16 keys (two 8-key tiles), 8 k-steps of 16 dims ----
            float sc[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                // matrices: (keys 0-7 | 8-15) x (dims 16ks..+7 | +8..+15)
                const int key = (lane & 7) + ((lane >> 4) & 1) * 8;
                const int chg = 2 * ks + ((lane >> 3) & 1);  // 16-byte chunk of the 128 dims
                uint32_t b0, b1, b2, b3;
                ldsm_x4(sa + (chg >> 3) * AD_BOX + ad_swz(key, chg & 7), b0, b1, b2, b3);
                const uint32_t a[4] = {qa[ks][0], 0u, qa[ks][1], 0u};
                mma16816(sc[0], a, b0, b1);
                mma16816(sc[1], a, b2, b3);
            }
            // ---- online softmax (exp2 domain) on this lane's row ----
            float mx = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = nt * 8 + 2 * tq + e;
                    sc[nt][e] = key < nvalid ? sc[nt][e] * p.scale_log2 : -INFINITY;
                    mx = fmaxf(mx, sc[nt][e]);
                }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mn = fmaxf(m_r, mx);
            const float alpha = (m_r == -INFINITY) ? 0.f : exp2f(m_r - mn);
            m_r = mn;
            float pv[2][2];
            float ls = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    pv[nt][e] = exp2f(sc[nt][e] - mn);
                    ls += pv[nt][e];
                }
            l_r = l_r * alpha + ls;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                o[nt][0] *= alpha;
                o[nt][1] *= alpha;
            }
            // P as the A operand of P V (rows 8-15 zero)
            const uint32_t pa[4] = {pack_h2(pv[0][0], pv[0][1]), 0u, pack_h2(pv[1][0], pv[1][1]), 0u};
            // ---- O += P V: 16 dims tiles of 8, keys 0-15 in one k-step ----
#pragma unroll
            for (int np = 0; np < 8; ++np) {
                const int key = (lane & 7) + ((lane >> 3) & 1) * 8;
                const int chg = 2 * np + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(sa + 2 * AD_BOX + (chg >> 3) * AD_BOX + ad_swz(key, chg & 7), b0, b1, b2, b3);
                mma16816(o[2 * np], pa, b0, b1);
                mma16816(o[2 * np + 1], pa, b2, b3);
            }
            __syncwarp();
            if (lane == 0) {
                // generic writes (the zeroed rows) before the next asynchronous refill
                if (nvalid < 16) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(ad_smem(empty + s)) : "memory");
            }
        }
        k_base += n;
        // row sums over the four lanes of a row group
        l_r += __shfl_xor_sync(0xffffffffu, l_r, 1);
        l_r += __shfl_xor_sync(0xffffffffu, l_r, 2);
        if (lane < 8) {
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                sm_o[(warp * 2 + gq) * 128 + nt * 8 + 2 * tq] = o[nt][0];
                sm_o[(warp * 2 + gq) * 128 + nt * 8 + 2 * tq + 1] = o[nt][1];
            }
            if (tq == 0) {
                sm_m[warp * 2 + gq] = m_r;
                sm_l[warp * 2 + gq] = l_r;
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(AD_CW * 32) : "memory");
        // threads 0..127 merge: (head hh, dims d2, d2 + 1)
        const int hh = (tid >> 6) & 1, d2 = (tid & 63) * 2;
        const bool merger = tid < 128;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < AD_CW; ++w) M = fmaxf(M, sm_m[w * 2 + hh]);
        float L = 0.f, O0 = 0.f, O1 = 0.f;
#pragma unroll
        for (int w = 0; w < AD_CW; ++w) {
            const float f = (sm_m[w * 2 + hh] == -INFINITY) ? 0.f : exp2f(sm_m[w * 2 + hh] - M);
            L += sm_l[w * 2 + hh] * f;
            O0 += sm_o[(w * 2 + hh) * 128 + d2] * f;
            O1 += sm_o[(w * 2 + hh) * 128 + d2 + 1] * f;
        }
        const int head = 2 * g + hh;
        f16* outp = p.out + ((size_t)t * p.n_heads + head) * 128 + d2;
        const int np = pref[t + 1] - pref[t];
        const long long pair0 = (long long)p.n_kv * pref[t] + (long long)g * np;
        if (i0 == 0 && n == np) {  // the whole pair is in this CTA
            if (merger) *reinterpret_cast<uint32_t*>(outp) = pack_h2(O0 / L, O1 / L);
        } else {
            const int cf = ad_cta_of(pair0, N, G);
            const int n_slots = ad_cta_of(pair0 + np - 1, N, G) - cf + 1;
            const size_t slot = ((size_t)t * p.n_heads + head) * p.max_slots + (c - cf);
            if (merger) {
                *reinterpret_cast<float2*>(p.part_o + slot * 128 + d2) = make_float2(O0, O1);
                if ((tid & 63) == 0) *reinterpret_cast<float2*>(p.part_ml + slot * 2) = make_float2(M, L);
            }
            // the CTA barrier orders every thread's partial before thread 0's fence, which
            // releases them (cumulatively) ahead of the ticket; the last CTA's thread 0
            // fences after the ticket (acquire) before the barrier that lets the merge read
            asm volatile("bar.sync 1, %0;" ::"n"(AD_CW * 32) : "memory");
            if (tid == 0) {
                __threadfence();
                const bool last = atomicAdd(p.counters + (size_t)t * p.n_kv + g, 1) == n_slots - 1;
                __threadfence();
                *last_flag = last;
            }
            asm volatile("bar.sync 1, %0;" ::"n"(AD_CW * 32) : "memory");
            if (*last_flag && merger) {
                const size_t base = ((size_t)t * p.n_heads + head) * p.max_slots;
                float MM = -INFINITY;
                for (int z = 0; z < n_slots; ++z) MM = fmaxf(MM, __ldcg(p.part_ml + (base + z) * 2));
                float LL = 0.f, A0 = 0.f, A1 = 0.f;
                for (int z = 0; z < n_slots; ++z) {
                    const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml + (base + z) * 2));
                    const float f = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - MM);
                    const float2 ov = __ldcg(reinterpret_cast<const float2*>(p.part_o + (base + z) * 128 + d2));
                    LL += ml.y * f;
                    A0 += ov.x * f;
                    A1 += ov.y * f;
                }
                *reinterpret_cast<uint32_t*>(outp) = pack_h2(A0 / LL, A1 / LL);
                if (tid == 0) p.counters[(size_t)t * p.n_kv + g] = 0;
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(AD_CW * 32) : "memory");  // shared merge buffers are reused
        j += n;
    }
}

int attn_decode_smem_bytes() { return AD_SMEM; }

cudaError_t launch_attn_decode(const LaunchCtx& c, int T, int layer, const f16* q, int n_heads, int n_kv, KVView kv,
                               const CUtensorMap* tmK, const CUtensorMap* tmV, const int* seqs, int max_keys,
                               int max_slots, float* part_o, float* part_ml, int* counters, f16* out, int* status,
                               int num_sms) {
    AttnDP p;
    memset(&p, 0, sizeof p);
    p.tmK = *tmK;
    p.tmV = *tmV;
    p.q = q;
    p.out = out;
    p.kv = kv;
    p.layer = layer;
    p.n_heads = n_heads;
    p.n_kv = n_kv;
    p.T = T;
    p.part_o = part_o;
    p.part_ml = part_ml;
    p.counters = counters;
    p.max_slots = max_slots;
    p.status = status;
    p.scale_log2 = 0.08838834764831845f * 1.4426950408889634f;  // 128^-0.5 * log2(e)
    for (int t = 0; t < T; ++t) p.seqp[t] = seqs[t];
    const int smem = attn_decode_smem_bytes();
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_attn_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    // at most one CTA per item; a pair spans at most G / n_kv + 2 CTAs (<= max_slots)
    const long long items = (long long)T * n_kv * ((max_keys + 15) / 16);
    int G = (int)std::min<long long>(2LL * num_sms, std::max(items, 1LL));
    G = std::min(G, (max_slots - 2) * n_kv);
    return launch_k(c, k_attn_decode, dim3(G), dim3(AD_THREADS), (size_t)smem, p);
}

// =======================================================================================
// k_attn_prefill_tc: causal GQA attention of a prefill on tcgen05 (Paso 5). A CTA takes 64
// queries of one sequence for both query heads 2g, 2g+1 of KV head g: the 128 rows of the MMA
// (rows 0-63 head 2g, 64-127 head 2g+1), so every K/V tile read from the cache serves both
// heads. Per tile of 64 keys, read from the sequence's cache pages with TMA (128-byte swizzle):
//   S = Q K^T     -> TMEM, two buffers, so the next tile's S overlaps this tile's softmax;
//   softmax       -> four warps, thread = row = TMEM lane, running max and sum in fp32 in the
//                    exp2 domain; P (fp16) goes back into the first half of its S buffer;
//   O += P V      -> A = P from TMEM, B = V as loaded ([key][dim], MN-major), O in TMEM.
// A row's running max moves only when a tile's max exceeds it by more than 2^8 (then O and
// the sum are rescaled), so most tiles skip the rescale and P stays <= 256; the final
// normalisation by the sum is exact either way. One thread issues the MMAs; one streams K and
// one V, each in a ring of two tiles that is released as soon as its MMA finished (K after
// S = Q K^T, V after O += P V), so the next K tile loads while this tile's softmax runs.
// 96 KB of shared memory and 256 TMEM columns let two CTAs share an SM; every wait is bounded.
// =======================================================================================
namespace {

constexpr int FA_BQ = 64;               // queries per head (128 MMA rows for the head pair)
constexpr int FA_BK = 64;               // keys per tile
constexpr int FA_THREADS = 224;         // warps 0-3 softmax/output, 4 K producer, 5 MMA, 6 V producer
constexpr int FA_QSUB = 128 * 128;      // Q: [128 rows][64 dims] swizzled subtile (16 KB)
constexpr int FA_KSUB = FA_BK * 128;    // K, V: [64 keys][64 dims] swizzled subtile (8 KB)
constexpr int FA_KV = 2 * FA_KSUB;      // one K or V tile, all 128 dims
constexpr int FA_OFF_K = 2 * FA_QSUB;   // [2] stages
constexpr int FA_OFF_V = FA_OFF_K + 2 * FA_KV;
constexpr int FA_OFF_BAR = FA_OFF_V + 2 * FA_KV;
constexpr int FA_SMEM = 1024 + FA_OFF_BAR + 256;
constexpr int FA_TMEM_COLS = 256;       // S[0] 0-63, S[1] 64-127, O 128-255
constexpr int FA_O = 128;
constexpr float FA_RESCALE_LOG2 = 8.f;  // the running max moves only past 2^8

__device__ __forceinline__ void fa_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

}  // namespace

struct PrefillTcP {
    CUtensorMap tmK;  // K pool as [n_layers * n_pages * n_kv * 16, 128] fp16
    CUtensorMap tmV;
    StepDesc sd;
    const f16* q;     // [T][n_heads][128]
    f16* out;         // [T][n_heads][128]
    const int* page_table;
    const int* tok_pos;  // [T] position of each token (a sequence's tokens continue its cache)
    int max_pages_per_seq, n_pages, layer, n_heads, n_kv;
    int* status;
    float scale_log2;
};

__global__ void __launch_bounds__(FA_THREADS, 2) k_attn_prefill_tc(const __grid_constant__ PrefillTcP p) {
    extern __shared__ uint8_t fa_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(fa_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + FA_OFF_BAR);
    uint64_t* k_full = bars;        // [2] K of a stage landed
    uint64_t* v_full = bars + 2;    // [2] V of a stage landed
    uint64_t* k_empty = bars + 4;   // [2] S = Q K^T of the stage finished
    uint64_t* v_empty = bars + 6;   // [2] O += P V of the stage finished
    uint64_t* s_full = bars + 8;    // [2] S buffer written
    uint64_t* p_full = bars + 10;   // [2] P written into the S buffer, O rescaled
    // [2] O += P V of the even / odd tiles finished. One barrier per tile parity: when a
    // softmax warp finishes its last tile, P V of the two previous tiles may still be pending,
    // and a single barrier's parity could not tell those three states apart.
    uint64_t* pv_done = bars + 12;
    uint64_t* q_ready = bars + 14;
    uint64_t* mma_fin = bars + 15;  // every MMA of the CTA finished (before TMEM is freed)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, g = blockIdx.y;
    const int len = p.sd.start[b + 1] - p.sd.start[b];
    const int q0 = ((int)gridDim.x - 1 - (int)blockIdx.x) * FA_BQ;  // heavy (late) query tiles first
    pdl_launch();
    if (q0 >= len) return;  // uniform over the CTA
    const int base = p.sd.start[b];
    auto wait = [&](uint64_t* bar, int parity) { return mbar_wait(smem_u32(bar), (uint32_t)parity & 1u, abort_flag); };

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(k_full + i), 1);
            mbar_init(smem_u32(v_full + i), 1);
            mbar_init(smem_u32(k_empty + i), 1);
            mbar_init(smem_u32(v_empty + i), 1);
            mbar_init(smem_u32(s_full + i), 1);
            mbar_init(smem_u32(p_full + i), 4);
            mbar_init(smem_u32(pv_done + i), 1);
        }
        mbar_init(smem_u32(q_ready), 4);
        mbar_init(smem_u32(mma_fin), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 4 && lane == 0) tma_prefetch_desc(&p.tmK);
    if (warp == 6 && lane == 0) tma_prefetch_desc(&p.tmV);
    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(FA_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();  // q and this layer's K/V come from the projection
    // The call's tokens of this sequence sit at positions L0 .. L0 + len - 1 after a cached
    // prefix of L0 tokens (0 for a first prompt); the keys are every position < L0 + len, and
    // query L0 + i sees keys <= L0 + i. This tile's queries need keys < L0 + min(len, q0 + 64).
    const int L0 = p.tok_pos[base];
    const int kend = L0 + len;
    const int n_kt = (L0 + min(len, q0 + FA_BQ) + FA_BK - 1) / FA_BK;

    if (warp == 4 || warp == 6) {
        // ---------------- producers: warp 4 streams K, warp 6 streams V ----------------
        if (lane == 0) {
            const bool is_k = warp == 4;
            const CUtensorMap* tm = is_k ? &p.tmK : &p.tmV;
            uint64_t* full = is_k ? k_full : v_full;
            uint64_t* empty = is_k ? k_empty : v_empty;
            uint8_t* ring = sm + (is_k ? FA_OFF_K : FA_OFF_V);
            const int* pt = p.page_table + (size_t)p.sd.seq[b] * p.max_pages_per_seq;
            const long long layer_rows = (long long)p.layer * p.n_pages;
            int issued = 0;
            for (int j = 0; j < n_kt && !*abort_flag; ++j, ++issued) {
                const int st = j & 1;
                if (j >= 2 && !wait(empty + st, (j >> 1) - 1)) {
                    *abort_flag = 1;
                    break;
                }
                const int k0 = j * FA_BK;
                const int npg = (min(k0 + FA_BK, kend) - k0 + 15) >> 4;
                const uint32_t dst = smem_u32(ring + st * FA_KV), bar = smem_u32(full + st);
                mbar_expect_tx(bar, (uint32_t)npg * 2 * 2048);
                for (int pg = 0; pg < npg; ++pg) {
                    const int pi = (k0 >> 4) + pg;
                    int page = pi < p.max_pages_per_seq ? pt[pi] : 0;
                    if (page < 0 || page >= p.n_pages) page = 0;  // bad pages were reported by the append
                    const int row = (int)(((layer_rows + page) * p.n_kv + g) * 16);
                    tma_load_2d(dst + pg * 2048, tm, bar, 0, row);
                    tma_load_2d(dst + FA_KSUB + pg * 2048, tm, bar, 64, row);
                }
            }
            // Before the CTA retires, the copies issued must have landed and the MMA thread's
            // releases of the last two tiles (asynchronous arrivals from tcgen05.commit) must have
            // reached this ring's barriers: an arrival still in flight would land in the shared
            // memory of the next CTA on this SM. At once on the normal path; bounded when another
            // role gave up.
            for (int jj = max(0, issued - 2); jj < issued; ++jj) {
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(smem_u32(full + (jj & 1)), (jj >> 1) & 1) && globaltimer_ns() - t0 < kTcWaitNs) {
                }
                while (!*abort_flag && !mbar_try_wait(smem_u32(empty + (jj & 1)), (jj >> 1) & 1) &&
                       globaltimer_ns() - t0 < kTcWaitNs) {
                }
            }
        }
    } else if (warp == 5) {
        // ---------------- MMA issuer: S_0, S_1, PV_0, S_2, PV_1, ... ----------------
        // S_{j+2} reuses the TMEM columns of S_j / P_j: it is issued only once PV_j, which
        // reads P_j from those columns, has finished (issue order alone does not keep a later
        // MMA's accumulator writes behind an earlier MMA's reads of A from tensor memory).
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_f16(128, FA_BK);
            constexpr uint32_t idesc_o = idesc_f16(128, 128) | kIdescBMajorMN;
            const uint32_t qa = smem_u32(sm);
            bool ok = wait(q_ready, 0);
            for (int j = 0; j <= n_kt && ok; ++j) {
                if (j < n_kt) {
                    const int st = j & 1;
                    if (!wait(k_full + st, j >> 1) || (j >= 2 && !wait(pv_done + st, (j - 2) >> 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ka = smem_u32(sm + FA_OFF_K + st * FA_KV);
#pragma unroll
                    for (int sub = 0; sub < 2; ++sub)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_f16(tmem + st * FA_BK, sw128_desc(qa + sub * FA_QSUB) + 2 * kk,
                                     sw128_desc(ka + sub * FA_KSUB) + 2 * kk, idesc_s, (sub | kk) ? 1u : 0u);
                    umma_commit(smem_u32(s_full + st));
                    umma_commit(smem_u32(k_empty + st));
                }
                if (j >= 1) {
                    const int jj = j - 1, sp = jj & 1;
                    if (!wait(p_full + sp, jj >> 1) || !wait(v_full + sp, jj >> 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t va = smem_u32(sm + FA_OFF_V + sp * FA_KV);
#pragma unroll
                    for (int kk = 0; kk < FA_BK / 16; ++kk)
                        umma_f16_ts(tmem + FA_O, tmem + sp * FA_BK + kk * 8, sw128_desc_mn(va + kk * 16 * 128, FA_KSUB),
                                    idesc_o, (jj | kk) ? 1u : 0u);
                    umma_commit(smem_u32(pv_done + sp));
                    umma_commit(smem_u32(v_empty + sp));
                }
            }
            if (!ok) *abort_flag = 1;
            umma_commit(smem_u32(mma_fin));
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(mma_fin), 0) && globaltimer_ns() - t0 < kTcWaitNs) {
            }
        }
    } else {
        // ---------------- softmax / output: thread = row = TMEM lane ----------------
        const int r = threadIdx.x;
        const int hq = 2 * g + (r >> 6), qi = q0 + (r & 63), qpos = L0 + qi;  // index in the call, position
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        // warp-uniform outcome of a bounded wait
        auto wwait = [&](uint64_t* bar, int parity) { return __all_sync(0xffffffffu, wait(bar, parity)); };
        {
            // Q row into the swizzled operand (zeros past the sequence)
            const bool v = qi < len;
            const f16* src = p.q + ((size_t)(base + (v ? qi : 0)) * p.n_heads + hq) * 128;
            const uint32_t qd = smem_u32(sm) + r * 128;
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) cp_async16(qd + (ch >> 3) * FA_QSUB + (((ch & 7) ^ (r & 7)) << 4), src + ch * 8, v);
            cp_commit();
            cp_wait<0>();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) fa_arrive(smem_u32(q_ready));
        }
        float m = -INFINITY, l = 0.f;
        bool good = true;
        for (int j = 0; j < n_kt; ++j) {
            const int st = j & 1, k0 = j * FA_BK;
            if (!wwait(s_full + st, j >> 1)) {
                good = false;
                break;
            }
            tc_fence_after();
            uint32_t xa[32], xb[32];
            TMEM_LD32(lane_base + st * FA_BK, xa);
            TMEM_LD32(lane_base + st * FA_BK + 32, xb);
            tmem_wait_ld();
            // raw scores q.k; the scale (> 0) is applied inside the exponent below
            float s[FA_BK];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                s[i] = __uint_as_float(xa[i]);
                s[32 + i] = __uint_as_float(xb[i]);
            }
            // mask keys after the query or past the sequence, on the tiles that hold any
            if (k0 + FA_BK - 1 > L0 + q0 || k0 + FA_BK > kend) {
#pragma unroll
                for (int i = 0; i < FA_BK; ++i)
                    if (k0 + i > qpos || k0 + i >= kend) s[i] = -INFINITY;
            }
            // row max through 8 independent partial maxima (short dependency chains)
            float pm[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) pm[u] = s[u];
#pragma unroll
            for (int i = 8; i < FA_BK; ++i) pm[i & 7] = fmaxf(pm[i & 7], s[i]);
            const float mt = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                                   fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7]))) * p.scale_log2;
            const bool move = mt > m + FA_RESCALE_LOG2;  // always on the first tile (m = -inf)
            const float mn = move ? mt : m;
            const float alpha = move ? ex2_approx(m - mn) : 1.f;  // 2^-inf = 0 on the first tile
            if (j > 0 && __any_sync(0xffffffffu, move)) {
                // O holds tiles < j at the old max: once P V of tile j-1 is done, rescale it
                if (!wwait(pv_done + ((j - 1) & 1), (j - 1) >> 1)) {
                    good = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t x[32];
                    TMEM_LD32(lane_base + FA_O + c * 32, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[i] = __float_as_uint(__uint_as_float(x[i]) * alpha);
                    TMEM_ST32(lane_base + FA_O + c * 32, x);
                }
            }
            float lp[4] = {0.f, 0.f, 0.f, 0.f};  // partial sums (short dependency chains)
            uint32_t h[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float e0 = ex2_approx(fmaf(s[2 * i], p.scale_log2, -mn));
                const float e1 = ex2_approx(fmaf(s[2 * i + 1], p.scale_log2, -mn));
                lp[i & 3] += e0 + e1;
                h[i] = pack_h2(e0, e1);
            }
            l = l * alpha + ((lp[0] + lp[1]) + (lp[2] + lp[3]));
            m = mn;
            TMEM_ST32(lane_base + st * FA_BK, h);
            if (j == n_kt - 1 && k0 + FA_BK > kend) {
                // V rows of keys past the sequence hold stale data; weight 0 must add exactly 0
                if (!wwait(v_full + st, j >> 1)) {
                    tmem_wait_st();
                    good = false;
                    break;
                }
                uint8_t* vs = sm + FA_OFF_V + st * FA_KV;
                const int kv0 = kend - k0;  // first row past the sequence
                for (int e = lane; e < 16 * 16; e += 32) {
                    const int row = warp * 16 + (e >> 4), ch = e & 15;
                    if (row >= kv0)
                        *reinterpret_cast<uint4*>(vs + (ch >> 3) * FA_KSUB + row * 128 + ((ch & 7) << 4)) =
                            make_uint4(0u, 0u, 0u, 0u);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) fa_arrive(smem_u32(p_full + st));
        }
        // ---- normalise and store the rows ----
        if (good && wwait(pv_done + ((n_kt - 1) & 1), (n_kt - 1) >> 1)) {
            tc_fence_after();
            const float inv = 1.f / l;
            f16* orow = p.out + ((size_t)(base + qi) * p.n_heads + hq) * 128;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t x[32];
                TMEM_LD32(lane_base + FA_O + c * 32, x);
                tmem_wait_ld();
                if (qi < len) {
                    uint32_t h[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        h[i] = pack_h2(__uint_as_float(x[2 * i]) * inv, __uint_as_float(x[2 * i + 1]) * inv);
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        *reinterpret_cast<uint4*>(orow + c * 32 + u * 8) = make_uint4(h[4 * u], h[4 * u + 1], h[4 * u + 2], h[4 * u + 3]);
                }
            }
        } else {
            *abort_flag = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) atomicOr(p.status, QW_DEV_TIMEOUT);
    if (warp == 5) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(FA_TMEM_COLS) : "memory");
    }
}

cudaError_t launch_attn_prefill_tc(const LaunchCtx& c, const StepDesc& sd, const int* tok_pos, int layer, const f16* q,
                                   KVView kv, const CUtensorMap* tmK, const CUtensorMap* tmV, int n_heads, int n_kv,
                                   f16* out, int* status) {
    PrefillTcP p;
    memset(&p, 0, sizeof p);
    p.tmK = *tmK;
    p.tmV = *tmV;
    p.sd = sd;
    p.q = q;
    p.out = out;
    p.page_table = kv.page_table;
    p.tok_pos = tok_pos;
    p.max_pages_per_seq = kv.max_pages_per_seq;
    p.n_pages = kv.n_pages;
    p.layer = layer;
    p.n_heads = n_heads;
    p.n_kv = n_kv;
    p.status = status;
    p.scale_log2 = 0.08838834764831845f * 1.4426950408889634f;  // 128^-0.5 * log2(e)
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_attn_prefill_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, FA_SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    int max_len = 1;
    for (int b = 0; b < sd.B; ++b) max_len = std::max(max_len, sd.start[b + 1] - sd.start[b]);
    const int qtiles = (max_len + FA_BQ - 1) / FA_BQ;
    return launch_k(c, k_attn_prefill_tc, dim3(qtiles, n_kv, sd.B), dim3(FA_THREADS), (size_t)FA_SMEM, p);
}
