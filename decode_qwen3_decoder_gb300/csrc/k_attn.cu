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
#include <utility>

#include "qw_internal.h"

namespace {

template <typename... KArgs, typename... Args>
cudaError_t launch_k(const LaunchCtx& c, void (*kern)(KArgs...), dim3 grid, dim3 block,
                     size_t smem, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[1];
    cfg.numAttrs = 0;
    if (c.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    if (c.counter) ++*c.counter;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

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
// k_attn_prefill: causal GQA attention of a prefill (sequences start empty, so position =
// index in the prompt) on the tensor cores, flash style (Paso 5): for each tile of 64
// queries of one sequence and one KV head, both query heads 2g and 2g+1 (128 rows, 8 warps
// of 16 rows) stream the sequence's K/V tiles of 64 keys through shared memory once.
// S = Q K^T and O += P V use mma.sync m16n8k16 (fp16 operands, fp32 accumulation); the
// online softmax runs in fp32 in the exp2 domain; P goes from the S accumulators straight
// into the A fragments of P V. K/V tiles (the new keys were just appended to the paged
// cache: key j sits at page_table[seq][j / 16], slot j % 16) are double-buffered with
// cp.async; shared rows of
// 256 bytes are XOR-swizzled by 16-byte chunk so ldmatrix is conflict-free. Key tiles past
// the query tile are skipped; the diagonal tile is masked key > query.
// =======================================================================================
namespace {

constexpr int PF_Q = 64;      // queries per CTA (per head)
constexpr int PF_KV = 64;     // keys per tile
constexpr int PF_WARPS = 8;

__device__ __forceinline__ uint32_t swz(int row, int chunk) {  // byte offset in a 256-byte-row tile
    return (uint32_t)(row * 256 + ((chunk ^ (row & 7)) << 4));
}
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

struct PrefillP {
    StepDesc sd;
    const f16* q;       // [T][n_heads][128]
    const f16* k;       // this layer's K pool [n_pages][n_kv][16][128]
    const f16* v;
    const int* page_table;
    int max_pages_per_seq, n_pages;
    f16* out;           // [T][n_heads * 128]
    int n_heads, n_kv;
    float scale_log2;
};

__global__ void __launch_bounds__(PF_WARPS * 32) k_attn_prefill(const __grid_constant__ PrefillP p) {
    extern __shared__ __align__(128) uint8_t pf_smem[];
    const uint32_t sQ = (uint32_t)__cvta_generic_to_shared(pf_smem);  // [128 rows][256 B]
    const uint32_t sK = sQ + 128 * 256;                               // [2][64][256 B]
    const uint32_t sV = sK + 2 * PF_KV * 256;                         // [2][64][256 B]
    pdl_launch();
    pdl_wait();
    const int b = blockIdx.z, g = blockIdx.y;
    const int len = p.sd.start[b + 1] - p.sd.start[b];
    const int qt = (int)gridDim.x - 1 - (int)blockIdx.x;  // heavy (late) query tiles first
    const int q0 = qt * PF_Q;
    if (q0 >= len) return;
    const int base = p.sd.start[b];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int* pt = p.page_table + (size_t)p.sd.seq[b] * p.max_pages_per_seq;

    // ---- Q tile: rows 0..63 head 2g, rows 64..127 head 2g+1 ---------------------------
    for (int i = tid; i < 128 * 16; i += PF_WARPS * 32) {
        const int row = i >> 4, ch = i & 15;
        const int hq = 2 * g + (row >> 6), qi = q0 + (row & 63);
        const bool v = qi < len;
        const f16* src = p.q + ((size_t)(base + (v ? qi : 0)) * p.n_heads + hq) * 128 + ch * 8;
        cp_async16(sQ + swz(row, ch), src, v);
    }
    auto load_kv = [&](int kt, int buf) {
        const int k0 = kt * PF_KV;
        // 256 threads x 4: pass j copies rows 16 j .. 16 j + 15 = page j of the tile
        static_assert(PF_KV == 64 && PF_WARPS * 32 == 256, "one page per pass");
        int page[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int pi = (k0 >> 4) + j;
            page[j] = (pi * 16 < len && pi < p.max_pages_per_seq) ? pt[pi] : -1;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int row = (tid >> 4) + 16 * j, ch = tid & 15;
            const int kj = k0 + row;  // key position (the sequence started empty)
            const bool v = kj < len && page[j] >= 0 && page[j] < p.n_pages;  // bad pages were reported
            const size_t off = (((size_t)(v ? page[j] : 0) * p.n_kv + g) * 16 + (kj & 15)) * 128 + ch * 8;
            cp_async16(sK + buf * PF_KV * 256 + swz(row, ch), p.k + off, v);
            cp_async16(sV + buf * PF_KV * 256 + swz(row, ch), p.v + off, v);
        }
    };
    const int n_kt = (min(len, q0 + PF_Q) + PF_KV - 1) / PF_KV;  // causal: keys < q0 + 64
    load_kv(0, 0);
    cp_commit();

    // this warp: 16 query rows of one head
    const int r0 = warp * 16;                   // row in the Q tile
    const int gq = lane >> 2, tq = lane & 3;
    const int qpos0 = q0 + (r0 & 63) + gq;      // positions of this thread's two rows
    const int qpos1 = qpos0 + 8;
    uint32_t qa[8][4];
    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int kt = 0; kt < n_kt; ++kt) {
        const int buf = kt & 1;
        if (kt + 1 < n_kt) load_kv(kt + 1, buf ^ 1);
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        if (kt == 0) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int row = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int ch = 2 * ks + (lane >> 4);
                ldsm_x4(sQ + swz(row, ch), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
            }
        }
        // ---- S = Q K^T (16 rows x 64 keys) ---------------------------------------------
        float s[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
        const uint32_t kb = sK + buf * PF_KV * 256;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
            for (int np = 0; np < 4; ++np) {  // pairs of 8-key n-tiles
                const int key = np * 16 + (lane & 7) + ((lane >> 4) & 1) * 8;
                const int ch = 2 * ks + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kb + swz(key, ch), b0, b1, b2, b3);
                mma16816(s[2 * np], qa[ks], b0, b1);
                mma16816(s[2 * np + 1], qa[ks], b2, b3);
            }
        }
        // ---- online softmax (exp2 domain), causal mask on the diagonal tile ---------------
        const int k0 = kt * PF_KV;
        float tm0 = -INFINITY, tm1 = -INFINITY;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int kp = k0 + n * 8 + 2 * tq;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const bool in = (kp + e) < len;
                s[n][e] = (in && kp + e <= qpos0) ? s[n][e] * p.scale_log2 : -INFINITY;
                s[n][2 + e] = (in && kp + e <= qpos1) ? s[n][2 + e] * p.scale_log2 : -INFINITY;
                tm0 = fmaxf(tm0, s[n][e]);
                tm1 = fmaxf(tm1, s[n][2 + e]);
            }
        }
        tm0 = fmaxf(tm0, __shfl_xor_sync(0xffffffffu, tm0, 1));
        tm0 = fmaxf(tm0, __shfl_xor_sync(0xffffffffu, tm0, 2));
        tm1 = fmaxf(tm1, __shfl_xor_sync(0xffffffffu, tm1, 1));
        tm1 = fmaxf(tm1, __shfl_xor_sync(0xffffffffu, tm1, 2));
        const float nm0 = fmaxf(m0, tm0), nm1 = fmaxf(m1, tm1);
        // rows with no visible key yet keep m = -inf; guard the rescale against inf - inf
        const float a0 = (nm0 == -INFINITY) ? 1.f : exp2f(m0 - nm0);
        const float a1 = (nm1 == -INFINITY) ? 1.f : exp2f(m1 - nm1);
        m0 = nm0;
        m1 = nm1;
        l0 *= a0;
        l1 *= a1;
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            o[n][0] *= a0;
            o[n][1] *= a0;
            o[n][2] *= a1;
            o[n][3] *= a1;
        }
        uint32_t pa[4][4];  // P as A fragments of P V, 4 k-steps of 16 keys
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const float e0 = (m0 == -INFINITY) ? 0.f : exp2f(s[n][0] - m0);
            const float e1 = (m0 == -INFINITY) ? 0.f : exp2f(s[n][1] - m0);
            const float e2 = (m1 == -INFINITY) ? 0.f : exp2f(s[n][2] - m1);
            const float e3 = (m1 == -INFINITY) ? 0.f : exp2f(s[n][3] - m1);
            l0 += e0 + e1;
            l1 += e2 + e3;
            pa[n >> 1][(n & 1) * 2 + 0] = pack_h2(e0, e1);
            pa[n >> 1][(n & 1) * 2 + 1] = pack_h2(e2, e3);
        }
        // ---- O += P V ------------------------------------------------------------------------
        const uint32_t vb = sV + buf * PF_KV * 256;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
            for (int np = 0; np < 8; ++np) {  // pairs of 8-dim n-tiles
                const int key = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int ch = 2 * np + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vb + swz(key, ch), b0, b1, b2, b3);
                mma16816(o[2 * np], pa[ks], b0, b1);
                mma16816(o[2 * np + 1], pa[ks], b2, b3);
            }
        }
        __syncthreads();  // the buffer is refilled two iterations later
    }
    cp_wait<0>();
    // ---- normalise and store -------------------------------------------------------------
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float i0 = 1.f / l0, i1 = 1.f / l1;
    const int hq = 2 * g + (r0 >> 6);
#pragma unroll
    for (int n = 0; n < 16; ++n) {
        const int d = n * 8 + 2 * tq;
        if (qpos0 < len)
            *reinterpret_cast<uint32_t*>(p.out + ((size_t)(base + qpos0) * p.n_heads + hq) * 128 + d) =
                pack_h2(o[n][0] * i0, o[n][1] * i0);
        if (qpos1 < len)
            *reinterpret_cast<uint32_t*>(p.out + ((size_t)(base + qpos1) * p.n_heads + hq) * 128 + d) =
                pack_h2(o[n][2] * i1, o[n][3] * i1);
    }
}

cudaError_t launch_attn_prefill(const LaunchCtx& c, const StepDesc& sd, int max_len, int layer, const f16* q,
                                KVView kv, int n_heads, int n_kv, f16* out) {
    PrefillP p;
    p.sd = sd;
    p.q = q;
    p.k = kv.k + (size_t)layer * kv.layer_stride;
    p.v = kv.v + (size_t)layer * kv.layer_stride;
    p.page_table = kv.page_table;
    p.max_pages_per_seq = kv.max_pages_per_seq;
    p.n_pages = kv.n_pages;
    p.out = out;
    p.n_heads = n_heads;
    p.n_kv = n_kv;
    p.scale_log2 = 0.08838834764831845f * 1.4426950408889634f;
    const int smem = 128 * 256 + 4 * PF_KV * 256;  // 96 KB
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_attn_prefill, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int qtiles = (max_len + PF_Q - 1) / PF_Q;
    return launch_k(c, k_attn_prefill, dim3(qtiles, n_kv, sd.B), dim3(PF_WARPS * 32), (size_t)smem, p);
}
