// Pieces shared by the tensor-core GEMM kernels (k_gemm.cu) and the batched decode-step
// kernel (k_step.cu): tile constants, the shared-memory budget of a GEMM configuration, the
// kernel parameters, and the epilogues that turn an accumulator tile (staged in shared memory
// as [token][row]) into the step's outputs -- per-head QK-norm + RoPE + KV append for the
// q|k|v projection, SiLU(gate) * up for the interleaved gate/up projection, and the residual
// loads of o_proj / down_proj.
//
// Included (after qw_internal.h and tc_sm103.cuh) by each translation unit that needs it; its
// definitions are in an anonymous namespace.
#pragma once

namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // 64 fp16 = 128 bytes = one swizzle row
constexpr int GEMM_THREADS = 192;     // cluster kernel: 4 epilogue warps, producer, MMA
constexpr int GEMM_TC_THREADS = 320;  // persistent kernel: 8 epilogue warps, producer, MMA


// Epilogue warpgroups: threads 0-127 (barrier 1) and, in the persistent kernel, 128-255
// (barrier 2); helpers index threads within their warpgroup.
__device__ __forceinline__ int epi_tid() { return threadIdx.x & 127; }
__device__ __forceinline__ void named_bar_epi() {
    asm volatile("bar.sync %0, 128;" ::"r"(1 + (threadIdx.x >> 7)) : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// address of the same shared variable in cluster CTA `rank`
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

constexpr int EP = 132;                   // pitch (floats) of the [token][128] staging tile
constexpr int E_BYTES = 32 * EP * 4;      // 32 tokens
constexpr int EPH = 136;                  // pitch (halves) of the fp16 staging tile (q|k|v heads)
constexpr int EH_BYTES = 32 * EPH * 2;
constexpr int SMEM_BUDGET = 227 * 1024;
// 1: the persistent GEMM runs on CTA pairs (tcgen05.mma.cta_group::2) wherever the tiles allow
#ifndef QW_GEMM_PAIR
#define QW_GEMM_PAIR 1
#endif

// NWG: epilogue warpgroups; BSPLIT: CTAs sharing the B tile (2 for the CTA-pair MMA, each
// CTA holding BN / 2 of its rows)
template <int BN, int EPI, int NWG, int BSPLIT = 1>
struct GemmCfg {
    static constexpr int A_BYTES = BM * BK * 2;  // 16 KB
    static constexpr int B_BYTES = BN / BSPLIT * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int NBUF = (2 * BN <= 512) ? 2 : 1;
    static constexpr int TMEM_COLS = NBUF * BN < 32 ? 32 : NBUF * BN;
    static constexpr int SBEST_WG = (EPI == EPI_ARGMAX) ? 4 * BN * 8 : 0;
    static constexpr int E_WG = (EPI == EPI_QKV_HEADS) ? EH_BYTES : (EPI == EPI_SILU_MUL) ? E_BYTES : 0;
    static constexpr int META_WG = (EPI == EPI_QKV_HEADS) ? 2 * BN * 4 : 0;  // tpos, tdst
    static constexpr int SBEST_BYTES = NWG * SBEST_WG;
    static constexpr int STAGE_E_BYTES = NWG * E_WG;
    static constexpr int NW_BYTES = (EPI == EPI_QKV_HEADS) ? 256 * 4 : 0;
    static constexpr int META_BYTES = NWG * META_WG;
    static constexpr int EXTRA = SBEST_BYTES + STAGE_E_BYTES + NW_BYTES + META_BYTES;
    static constexpr int BAR_BYTES = 256;
    static constexpr int STAGES_RAW = (SMEM_BUDGET - 1024 - BAR_BYTES - EXTRA) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + EXTRA + BAR_BYTES;
};

struct GemmKParams {
    int a_row0, b_row0, K, T, ld_out;
    int tiles_m, tiles_n, units, splits;
    float* out_f32;  // EPI_RESID_F32: x [T][ld_out]
    f16* out_h;      // EPI_SILU_MUL: act [T][ld_out]
    float* logits;   // EPI_ARGMAX: optional [T][ld_out]
    unsigned long long* best;
    int* status;
    // EPI_QKV_HEADS
    f16* q_out;
    const bf16* q_norm;
    const bf16* k_norm;
    float eps;
    const float* rope_cos;
    const float* rope_sin;
    TokView tv;
    KVView kv;
    int layer, n_heads, n_kv;
    int32_t* dbg_pos;
    int32_t* dbg_slot;
};

// ---- epilogues over a staged [token][EP] fp32 tile (128 epilogue threads) -------------

// Token metadata of a q|k|v tile, filled while its MMAs run: tpos[c] = position of token
// n0 + c, tdst[c] = its KV slot row page * 16 + pos % 16 (-1: no page; reported), both
// computed once per step by the step's first kernel.
template <int BN>
__device__ void fill_tok_meta(const GemmKParams& p, int n0, int hd, int* tpos, int* tdst) {
    for (int c = epi_tid(); c < BN; c += 128) {
        const int tok = n0 + c;
        int pos = 0, dst = -1;
        if (tok < p.T) {
            pos = p.tv.pos[tok];
            dst = p.tv.slot[tok];
            if (dst < 0 && hd >= p.n_heads) atomicOr(p.status, QW_DEV_BAD_POS);
            if (p.dbg_pos && hd == p.n_heads) {
                p.dbg_pos[tok] = pos;
                p.dbg_slot[tok] = dst;
            }
        }
        tpos[c] = pos;
        tdst[c] = dst;
    }
}

// Head-epilogue thread layout over a staged chunk of 32 tokens: warp w of the warpgroup takes
// tokens 8w .. 8w + 7; lane l holds token t = 8w + l / 4 and quarter q = l % 4, i.e. the dims
// [16q, 16q + 16) of the head and their rotate-half partners 64 + 16q .. (the four quarters of
// a token are adjacent lanes, so the head's sum of squares needs two shuffles). The fp16
// staging rows have a pitch of 136 halves, so the 16-byte reads of 8 consecutive lanes hit
// distinct banks; every store is a whole 32-byte sector.
__device__ __forceinline__ int head_tok() { return ((epi_tid() >> 5) << 3) + ((threadIdx.x & 31) >> 2); }
__device__ __forceinline__ int head_qtr() { return threadIdx.x & 3; }

// RoPE cos/sin of this thread's 16 dims for its token (tpos[cbase + t]).
struct RopeRegs {
    float4 c[4], s[4];
};
__device__ __forceinline__ void load_rope(const GemmKParams& p, const int* tpos, int cbase, int ntok, RopeRegs& rr) {
    const int t = head_tok(), q = head_qtr();
    const int pos = t < ntok ? tpos[cbase + t] : 0;
    const float4* cs = reinterpret_cast<const float4*>(p.rope_cos + (size_t)pos * 64 + 16 * q);
    const float4* sn = reinterpret_cast<const float4*>(p.rope_sin + (size_t)pos * 64 + 16 * q);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        rr.c[k] = __ldg(cs + k);
        rr.s[k] = __ldg(sn + k);
    }
}

__device__ __forceinline__ void store16h(f16* dst, const float* v) {  // 16 values -> 32 bytes
    uint4 a, b;
    a.x = pack_h2(v[0], v[1]);
    a.y = pack_h2(v[2], v[3]);
    a.z = pack_h2(v[4], v[5]);
    a.w = pack_h2(v[6], v[7]);
    b.x = pack_h2(v[8], v[9]);
    b.y = pack_h2(v[10], v[11]);
    b.z = pack_h2(v[12], v[13]);
    b.w = pack_h2(v[14], v[15]);
    reinterpret_cast<uint4*>(dst)[0] = a;
    reinterpret_cast<uint4*>(dst)[1] = b;
}

// q|k|v head tile `hd`, tokens tok0 .. tok0 + ntok - 1 (tile columns cbase ..). q and k
// heads: RMSNorm over the head's 128 dims with the shared weight, then the rotation by
// pos * theta^(-i/64); v heads: copied.
__device__ void epi_heads(const GemmKParams& p, const f16* EH, const float* nws, const int* tdst,
                          const RopeRegs& rr, int tok0, int cbase, int ntok, int hd) {
    const int t = head_tok(), q = head_qtr();
    const bool isq = hd < p.n_heads;
    const bool isv = hd >= p.n_heads + p.n_kv;
    const f16* row = EH + t * EPH;  // the tile staged as fp16 [token][EPH]
    float a[16], b[16];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint4 va = *reinterpret_cast<const uint4*>(row + 16 * q + 8 * k);
        const uint4 vb = *reinterpret_cast<const uint4*>(row + 64 + 16 * q + 8 * k);
        const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            a[8 * k + 2 * i] = h_lo(wa[i]);
            a[8 * k + 2 * i + 1] = h_hi(wa[i]);
            b[8 * k + 2 * i] = h_lo(wb[i]);
            b[8 * k + 2 * i + 1] = h_hi(wb[i]);
        }
    }
    {
        // the tile was staged as fp16: a projection beyond the fp16 range is inf here
        bool big = false;
#pragma unroll
        for (int k = 0; k < 16; ++k) big |= f16_out_of_range(a[k]) || f16_out_of_range(b[k]);
        if (big && t < ntok) atomicOr(p.status, QW_DEV_RANGE);
    }
    if (!isv) {
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) ss = fmaf(a[k], a[k], fmaf(b[k], b[k], ss));
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        const float r = rsqrtf(ss * (1.0f / 128.0f) + p.eps);
        const float4* w4 = reinterpret_cast<const float4*>(nws + (isq ? 0 : 128) + 16 * q);
        float wa[16], wb[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 x = w4[k], y = w4[16 + k];  // dims 16q + 4k .. and 64 + 16q + 4k ..
            wa[4 * k] = x.x; wa[4 * k + 1] = x.y; wa[4 * k + 2] = x.z; wa[4 * k + 3] = x.w;
            wb[4 * k] = y.x; wb[4 * k + 1] = y.y; wb[4 * k + 2] = y.z; wb[4 * k + 3] = y.w;
        }
        const float c[16] = {rr.c[0].x, rr.c[0].y, rr.c[0].z, rr.c[0].w, rr.c[1].x, rr.c[1].y, rr.c[1].z, rr.c[1].w,
                             rr.c[2].x, rr.c[2].y, rr.c[2].z, rr.c[2].w, rr.c[3].x, rr.c[3].y, rr.c[3].z, rr.c[3].w};
        const float sn[16] = {rr.s[0].x, rr.s[0].y, rr.s[0].z, rr.s[0].w, rr.s[1].x, rr.s[1].y, rr.s[1].z, rr.s[1].w,
                              rr.s[2].x, rr.s[2].y, rr.s[2].z, rr.s[2].w, rr.s[3].x, rr.s[3].y, rr.s[3].z, rr.s[3].w};
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float ya = a[k] * r * wa[k], yb = b[k] * r * wb[k];
            a[k] = ya * c[k] - yb * sn[k];
            b[k] = yb * c[k] + ya * sn[k];
        }
    }
    if (t >= ntok) return;
    f16* dst;
    if (isq) {
        dst = p.q_out + ((size_t)(tok0 + t) * p.n_heads + hd) * 128;
    } else {
        const int slot = tdst[cbase + t];
        if (slot < 0) return;
        const int g = hd - p.n_heads - (isv ? p.n_kv : 0);
        dst = (isv ? p.kv.v : p.kv.k) + (size_t)p.layer * p.kv.layer_stride +
              (((size_t)(slot >> 4) * p.n_kv + g) * 16 + (slot & 15)) * 128;
    }
    store16h(dst + 16 * q, a);
    store16h(dst + 64 + 16 * q, b);
}

// SwiGLU thread layout: lane = token t of the chunk, warp q of the warpgroup = gate features
// [16q, 16q + 16) and the matching up rows.
// interleaved gate/up tile `tile` (gate rows 0..63, up rows 64..127 of output features
// 64 tile .. 64 tile + 63): act = SiLU(gate) * up.
__device__ void epi_silu(const GemmKParams& p, const float* E, int tok0, int ntok, int tile) {
    const int t = threadIdx.x & 31, q = epi_tid() >> 5;
    if (t >= ntok) return;
    const float* row = E + t * EP;
    float v[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float4 g = *reinterpret_cast<const float4*>(row + 16 * q + 4 * k);
        const float4 u = *reinterpret_cast<const float4*>(row + 64 + 16 * q + 4 * k);
        // fast exponential and division: their fp32 error is far below the fp16 rounding of act
        v[4 * k] = __fdividef(g.x, 1.0f + __expf(-g.x)) * u.x;
        v[4 * k + 1] = __fdividef(g.y, 1.0f + __expf(-g.y)) * u.y;
        v[4 * k + 2] = __fdividef(g.z, 1.0f + __expf(-g.z)) * u.z;
        v[4 * k + 3] = __fdividef(g.w, 1.0f + __expf(-g.w)) * u.w;
    }
    bool big = false;
#pragma unroll
    for (int k = 0; k < 16; ++k) big |= f16_out_of_range(v[k]);
    if (big) atomicOr(p.status, QW_DEV_RANGE);
    store16h(p.out_h + (size_t)(tok0 + t) * p.ld_out + tile * 64 + 16 * q, v);
}

// fp32 residual x[tok0 + j][f], j < 32 (0 past the last token)
__device__ __forceinline__ void load_resid(const GemmKParams& p, int tok0, int f, float* xr) {
#pragma unroll
    for (int j = 0; j < 32; ++j) xr[j] = (tok0 + j < p.T) ? __ldcg(p.out_f32 + (size_t)(tok0 + j) * p.ld_out + f) : 0.f;
}

__device__ __forceinline__ void load_norm_weights(const GemmKParams& p, float* nws) {
    for (int i = epi_tid(); i < 256; i += 128) nws[i] = __bfloat162float(i < 128 ? p.q_norm[i] : p.k_norm[i - 128]);
}

}  // namespace
