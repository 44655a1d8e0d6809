// Bandwidth-bound kernels of the decoder step: step bookkeeping + embedding gather,
// RMSNorm, the small-batch GEMV family (RMSNorm fused in the prologue), QK-norm + RoPE +
// paged KV append, the argmax finalize, and the synthetic KV fill.
//
// Page: "Dentro de un LLM: Inferencia en Python puro para Qwen3-0.6B en MLX".
#include <utility>

#include "qw_internal.h"

namespace {

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// 8 bf16 weights (one 16-byte chunk, widened exactly by a shift) against 8 fp32 activations.
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

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

}  // namespace

// =======================================================================================
// Step begin: embedding gather (Paso 2) + per-token sequence/position bookkeeping (Paso 9:
// positions continue from the sequence's current length).
// =======================================================================================
// ss (optional): per token, the sum of squares of x over each 128-feature block
// [t][hidden / 128], and xw = fp16(x * nw) [t][hidden] with nw the first layer's input-norm
// weight (the batched decode-step kernel builds its first RMSNorm from these).
__global__ void __launch_bounds__(256) k_step_begin(StepDesc sd, const int32_t* __restrict__ ids,
                                                    const bf16* __restrict__ embed, int vocab,
                                                    int hidden, float* __restrict__ x, TokView tv,
                                                    KVView kv, int* status, float* __restrict__ ss,
                                                    const bf16* __restrict__ nw, f16* __restrict__ xw) {
    // dependents start after the wait: what they read before their own wait (cached lengths,
    // page tables, K/V) is then complete even when this kernel was launched early
    pdl_wait();
    pdl_launch();
    const int t = blockIdx.x;
    int b = 0;
    while (b + 1 < sd.B && sd.start[b + 1] <= t) ++b;
    const int id = ids[t];
    const bool bad = (id < 0) || (id >= vocab);
    const bf16* src = embed + (size_t)(bad ? 0 : id) * hidden;
    float* dst = x + (size_t)t * hidden;
    for (int k = threadIdx.x * 4; k < hidden; k += blockDim.x * 4) {
        uint2 w = *reinterpret_cast<const uint2*>(src + k);
        float4 o = bad ? make_float4(0.f, 0.f, 0.f, 0.f)
                       : make_float4(bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y));
        *reinterpret_cast<float4*>(dst + k) = o;
        if (ss) {  // a warp covers the 128 features of block k / 128
            const float q = warp_sum(o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w);
            if ((threadIdx.x & 31) == 0) ss[(size_t)t * (hidden / 128) + k / 128] = q;
            const uint2 wv = *reinterpret_cast<const uint2*>(nw + k);
            uint2 h;
            h.x = pack_h2(o.x * bf_lo(wv.x), o.y * bf_hi(wv.x));
            h.y = pack_h2(o.z * bf_lo(wv.y), o.w * bf_hi(wv.y));
            *reinterpret_cast<uint2*>(xw + (size_t)t * hidden + k) = h;
        }
    }
    if (threadIdx.x == 0) {
        const int seq = sd.seq[b];
        const int pos = kv.len[seq] + (t - sd.start[b]);
        tv.seq[t] = seq;
        tv.pos[t] = pos;
        // the token's KV slot, the same for every layer (kernels that append report a missing page)
        const int pi = pos >> 4;
        const int page = (pi < kv.max_pages_per_seq) ? kv.page_table[(size_t)seq * kv.max_pages_per_seq + pi] : -1;
        tv.slot[t] = (page >= 0 && page < kv.n_pages) ? page * 16 + (pos & 15) : -1;
        if (t == sd.start[b + 1] - 1) tv.last[b] = t;
        if (bad) atomicOr(status, QW_DEV_BAD_TOKEN);
    }
}

cudaError_t launch_step_begin(const LaunchCtx& c, const StepDesc& sd, const int32_t* ids,
                              const bf16* embed, int vocab, int hidden, float* x, TokView tv,
                              KVView kv, int* status, float* ss, const bf16* w, f16* xw) {
    return launch_k(c, k_step_begin, dim3(sd.T), dim3(256), 0, sd, ids, embed, vocab, hidden, x, tv,
                    kv, status, ss, w, xw);
}

// =======================================================================================
// RMSNorm (Paso 3) of fp32 rows into fp16 GEMM operands: h = x * rsqrt(mean(x^2) + eps) * w.
// One warp per row; `rows` optionally gathers (the LM head reads each sequence's last row).
// =======================================================================================
__global__ void __launch_bounds__(256) k_rmsnorm(const float* __restrict__ x, const int* __restrict__ rows,
                                                 int n_rows, int hidden, const bf16* __restrict__ w,
                                                 float eps, f16* __restrict__ h) {
    pdl_launch();
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    // the norm weights are constant: requested before the dependency wait
    uint2 wv[8];
    if (hidden == 1024) {
#pragma unroll
        for (int u = 0; u < 8; ++u) wv[u] = *reinterpret_cast<const uint2*>(w + lane * 4 + u * 128);
    }
    pdl_wait();
    if (r < n_rows && hidden == 1024) {
        // the model's width: the row's 8 float4 per lane are requested together and kept in
        // registers (one round trip, no second read)
        const float* xr = x + (size_t)(rows ? rows[r] : r) * 1024;
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = *reinterpret_cast<const float4*>(xr + lane * 4 + u * 128);
        float ss = 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) ss += v[u].x * v[u].x + v[u].y * v[u].y + v[u].z * v[u].z + v[u].w * v[u].w;
        const float rs = rsqrtf(warp_sum(ss) / 1024.f + eps);
        f16* hr = h + (size_t)r * 1024;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int k = lane * 4 + u * 128;
            const uint2 wb = wv[u];
            uint2 o;
            o.x = pack_h2(v[u].x * rs * bf_lo(wb.x), v[u].y * rs * bf_hi(wb.x));
            o.y = pack_h2(v[u].z * rs * bf_lo(wb.y), v[u].w * rs * bf_hi(wb.y));
            *reinterpret_cast<uint2*>(hr + k) = o;
        }
    } else if (r < n_rows) {
        const float* xr = x + (size_t)(rows ? rows[r] : r) * hidden;
        float ss = 0.f;
        for (int k = lane * 4; k < hidden; k += 128) {
            float4 v = *reinterpret_cast<const float4*>(xr + k);
            ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
        const float rs = rsqrtf(warp_sum(ss) / (float)hidden + eps);
        f16* hr = h + (size_t)r * hidden;
        for (int k = lane * 4; k < hidden; k += 128) {
            float4 v = *reinterpret_cast<const float4*>(xr + k);
            uint2 wb = *reinterpret_cast<const uint2*>(w + k);
            uint2 o;
            o.x = pack_h2(v.x * rs * bf_lo(wb.x), v.y * rs * bf_hi(wb.x));
            o.y = pack_h2(v.z * rs * bf_lo(wb.y), v.w * rs * bf_hi(wb.y));
            *reinterpret_cast<uint2*>(hr + k) = o;
        }
    }
}

cudaError_t launch_rmsnorm(const LaunchCtx& c, const float* x, const int* rows, int n_rows,
                           int hidden, const bf16* w, float eps, f16* h) {
    return launch_k(c, k_rmsnorm, dim3((n_rows + 7) / 8), dim3(256), 0, x, rows, n_rows, hidden, w,
                    eps, h);
}

// =======================================================================================
// GEMV family for T <= 8 token rows: out[t][n] = sum_k W[n][k] * a[t][k].
//
// Each warp owns RPW output rows at a time; every lane streams one 16-byte chunk of each
// row per 256 columns, so a warp reads whole rows with coalesced 512-byte requests, in
// passes of 1024 columns that keep RPW*4 16-byte loads per lane in flight. The activations sit in
// shared memory as fp32; weights are the bf16 originals. MODE selects the prologue/epilogue:
//   G_QKV    : a = rms_norm(x) * w_in  (Paso 3 fused), out fp32 (Paso 5 projections)
//   G_GATEUP : a = rms_norm(x) * w_post, act = fp16(silu(Wg a) * (Wu a))  (Paso 6)
//   G_RESID  : a = fp16 activations, x += W a  (o_proj / down_proj + residual, Paso 7)
//   G_LMHEAD : a = rms_norm(x[last]) * w_final, logits, packed argmax (Paso 8)
// =======================================================================================
enum { G_QKV = 0, G_GATEUP = 1, G_RESID = 2, G_LMHEAD = 3 };

struct GemvP {
    const float* x;
    const int* rows;
    const bf16* norm_w;
    float eps;
    const f16* act;
    const bf16* W;
    const bf16* W2;
    // quantized weights (QB = 8 or 4): codes and per-group (scale, bias) half2 words
    const uint8_t* qw;
    const uint8_t* qw2;
    const uint32_t* sb;
    const uint32_t* sb2;
    int n_out;
    int K;
    int T;
    float* out;
    f16* out_h;
    unsigned long long* best;
    int* status;  // G_GATEUP: QW_DEV_RANGE when an fp16 activation would overflow
    // optional o_proj partial sums not yet in x: the residual seen by this kernel is
    // x + sum_g xadd[g][t][:] (g < n_add, added in order); G_GATEUP and G_RESID
    const float* xadd;
    int n_add;
};

constexpr int GEMV_WARPS = 4;

// Streaming 16-byte load issued in program order (volatile), so the weight fetches of a
// launch stay ahead of its griddepcontrol.wait.
__device__ __forceinline__ uint4 ldg_stream_v(const void* ptr) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(ptr));
    return r;
}
__device__ __forceinline__ uint2 ldg_stream_v2(const void* ptr) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(ptr));
    return r;
}
__device__ __forceinline__ uint32_t ldg_stream_u32(const void* ptr) {
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(ptr));
    return r;
}

// Eight dequantized weights (scale * q + bias) times eight activations: w.x (and w.y for
// 8-bit codes) hold the codes, w.z the group's (scale, bias) half2 word.
// A code c < 2^23 becomes a float exactly as (the float with bits 0x4B000000 | c) - 2^23:
// that float is 2^23 + c, so a logic op and one addition replace an int-to-float conversion.
__device__ __forceinline__ float code_to_float(uint32_t c) { return __uint_as_float(0x4B000000u | c) - 8388608.0f; }

// sa: the sum of the eight activations (the bias term's factor, shared by every row).
template <int QB>
__device__ __forceinline__ float dot8q(const uint4 w, const float4 a0, const float4 a1, float sa, float acc) {
    float q[8];
    if (QB == 8) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            q[i] = code_to_float((w.x >> (8 * i)) & 0xFFu);
            q[4 + i] = code_to_float((w.y >> (8 * i)) & 0xFFu);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = code_to_float((w.x >> (4 * i)) & 0xFu);
    }
    const float s = h_lo(w.z), b = h_hi(w.z);
    float dq = q[0] * a0.x;
    dq = fmaf(q[1], a0.y, dq);
    dq = fmaf(q[2], a0.z, dq);
    dq = fmaf(q[3], a0.w, dq);
    dq = fmaf(q[4], a1.x, dq);
    dq = fmaf(q[5], a1.y, dq);
    dq = fmaf(q[6], a1.z, dq);
    dq = fmaf(q[7], a1.w, dq);
    return fmaf(s, dq, fmaf(b, sa, acc));
}

// Programmatic dependent launch: the kernel lets its dependents launch at entry and issues
// the weight loads of its first row group before griddepcontrol.wait, so the weights (which
// no earlier kernel writes) stream from HBM while the upstream kernel is still finishing.
// Everything that reads upstream outputs, or writes anything, comes after the wait.
// QB: weight format, 16 = the bf16 originals, 8 / 4 = grouped affine codes (groups of 64).
template <int TT, int MODE, int KC, int RPW, int QB>
__global__ void __launch_bounds__(GEMV_WARPS * 32) k_gemv(GemvP p) {
    extern __shared__ float4 smem_f4[];
    float* hs = reinterpret_cast<float*>(smem_f4);  // [TT][K] fp32
    constexpr int K = KC * 256;
    constexpr int NW = (MODE == G_GATEUP) ? 2 : 1;
    constexpr int PC = (KC <= 12) ? KC : 4;  // 16-byte chunks per lane held per pass
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gw = blockIdx.x * GEMV_WARPS + warp;
    const int nw = gridDim.x * GEMV_WARPS;
    pdl_launch();

    uint4 wv[RPW][NW][PC];
    auto load_pass = [&](int r0, int c0) {
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const int row = min(r0 + rr, p.n_out - 1);
#pragma unroll
            for (int c = 0; c < PC; ++c) {
                const size_t off = (size_t)row * K + (c0 + c) * 256 + lane * 8;
                if (QB == 16) {
                    wv[rr][0][c] = ldg_stream_v(p.W + off);
                    if (NW == 2) wv[rr][NW - 1][c] = ldg_stream_v(p.W2 + off);
                } else {
                    const size_t gi = off / 64;  // group of these 8 inputs
#pragma unroll
                    for (int n = 0; n < NW; ++n) {
                        const uint8_t* cw = n ? p.qw2 : p.qw;
                        const uint32_t* sw = n ? p.sb2 : p.sb;
                        uint4 v;
                        if (QB == 8) {
                            const uint2 t = ldg_stream_v2(cw + off);
                            v.x = t.x;
                            v.y = t.y;
                        } else {
                            v.x = ldg_stream_u32(cw + off / 2);
                            v.y = 0u;
                        }
                        v.z = ldg_stream_u32(sw + gi);
                        v.w = 0u;
                        wv[rr][n][c] = v;
                    }
                }
            }
        }
    };
    if (gw * RPW < p.n_out) load_pass(gw * RPW, 0);
    // the RMSNorm weight slice of this thread is constant too: also before the wait
    constexpr int NCH = K / 512;  // float4 chunks of a row per thread (norm prologue)
    uint2 nwv[NCH > 0 ? NCH : 1];
    if (MODE != G_RESID) {
#pragma unroll
        for (int c = 0; c < NCH; ++c) nwv[c] = *reinterpret_cast<const uint2*>(p.norm_w + (tid + c * 128) * 4);
    }
    pdl_wait();

    // ---- prologue: activations into shared memory --------------------------------------
    float xres[RPW];  // G_RESID: residual x[token = lane][row] of this warp's first rows
    if (MODE == G_RESID) {
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const int row = gw * RPW + rr;
            float v = 0.f;
            if (lane < p.T && row < p.n_out) {
                v = p.out[(size_t)lane * p.n_out + row];
                for (int g = 0; g < p.n_add; ++g) v += p.xadd[((size_t)g * p.T + lane) * p.n_out + row];
            }
            xres[rr] = v;
        }
        for (int i = tid; i < TT * K / 8; i += blockDim.x) {
            const int t = i / (K / 8), k8 = (i % (K / 8)) * 8;
            float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
            if (t < p.T) {
                uint4 w = *reinterpret_cast<const uint4*>(p.act + (size_t)t * K + k8);
                a0 = make_float4(h_lo(w.x), h_hi(w.x), h_lo(w.y), h_hi(w.y));
                a1 = make_float4(h_lo(w.z), h_hi(w.z), h_lo(w.w), h_hi(w.w));
            }
            *reinterpret_cast<float4*>(hs + t * K + k8) = a0;
            *reinterpret_cast<float4*>(hs + t * K + k8 + 4) = a1;
        }
    } else {
        // one read of x: each thread stores its chunks of every token row raw into shared
        // memory while summing their squares; the sums meet in shared memory, then each
        // thread rescales its own chunks to h = x * rsqrt(mean(x^2) + eps) * w
        static_assert(K % 512 == 0, "norm prologue: 128 threads x float4 chunks");
        __shared__ float red[GEMV_WARPS][TT];
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            float part = 0.f;
            const bool live = t < p.T;
            const float* xr = p.x + (size_t)(live ? (p.rows ? p.rows[t] : t) : 0) * K;
            // every x load of the row first (unconditional: row 0 stands in for a dead row), so
            // that they are in flight together
            float4 v[NCH > 0 ? NCH : 1];
#pragma unroll
            for (int c = 0; c < NCH; ++c) v[c] = *reinterpret_cast<const float4*>(xr + (tid + c * 128) * 4);
            if (live && p.n_add) {  // o_proj partials not yet in x (decode rows: row t is token t)
                constexpr int GB = NCH <= 2 ? 8 : (NCH <= 4 ? 4 : 1);  // partials in flight per batch
                for (int g0 = 0; g0 < p.n_add; g0 += GB) {
                    // GB partials' loads in flight (indices clamped), added in order of g
                    float4 a[GB][NCH > 0 ? NCH : 1];
#pragma unroll
                    for (int j = 0; j < GB; ++j) {
                        const int g = min(g0 + j, p.n_add - 1);
#pragma unroll
                        for (int c = 0; c < NCH; ++c)
                            a[j][c] = *reinterpret_cast<const float4*>(p.xadd + ((size_t)g * p.T + t) * K + (tid + c * 128) * 4);
                    }
#pragma unroll
                    for (int j = 0; j < GB; ++j) {
                        if (g0 + j < p.n_add) {
#pragma unroll
                            for (int c = 0; c < NCH; ++c) {
                                v[c].x += a[j][c].x;
                                v[c].y += a[j][c].y;
                                v[c].z += a[j][c].z;
                                v[c].w += a[j][c].w;
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                if (!live) v[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4*>(hs + t * K + (tid + c * 128) * 4) = v[c];
                part += v[c].x * v[c].x + v[c].y * v[c].y + v[c].z * v[c].z + v[c].w * v[c].w;
            }
            part = warp_sum(part);
            if (lane == 0) red[warp][t] = part;
        }
        __syncthreads();
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            float ss = 0.f;
#pragma unroll
            for (int w = 0; w < GEMV_WARPS; ++w) ss += red[w][t];
            const float r = rsqrtf(ss / (float)K + p.eps);
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                float4* hp = reinterpret_cast<float4*>(hs + t * K + (tid + c * 128) * 4);
                const float4 v = *hp;
                const uint2 wb = nwv[c];
                *hp = make_float4(v.x * r * bf_lo(wb.x), v.y * r * bf_hi(wb.x), v.z * r * bf_lo(wb.y),
                                  v.w * r * bf_hi(wb.y));
            }
        }
    }
    __syncthreads();

    // ---- main loop ---------------------------------------------------------------------
    unsigned long long best[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) best[t] = 0ull;

    bool first = true, first_rows = true;
    for (int r0 = gw * RPW; r0 < p.n_out; r0 += nw * RPW) {
        float acc[RPW][NW][TT];
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr)
#pragma unroll
            for (int n = 0; n < NW; ++n)
#pragma unroll
                for (int t = 0; t < TT; ++t) acc[rr][n][t] = 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < KC; c0 += PC) {
            if (!first) load_pass(r0, c0);
            first = false;
#pragma unroll
            for (int c = 0; c < PC; ++c) {
#pragma unroll
                for (int t = 0; t < TT; ++t) {
                    const float* a = hs + t * K + (c0 + c) * 256 + lane * 8;
                    const float4 a0 = *reinterpret_cast<const float4*>(a);
                    const float4 a1 = *reinterpret_cast<const float4*>(a + 4);
                    const float sa = QB == 16 ? 0.f : ((a0.x + a0.y) + (a0.z + a0.w)) + ((a1.x + a1.y) + (a1.z + a1.w));
#pragma unroll
                    for (int rr = 0; rr < RPW; ++rr)
#pragma unroll
                        for (int n = 0; n < NW; ++n)
                            acc[rr][n][t] = QB == 16 ? dot8(wv[rr][n][c], a0, a1, acc[rr][n][t])
                                                     : dot8q<QB>(wv[rr][n][c], a0, a1, sa, acc[rr][n][t]);
                }
            }
        }
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const int row = r0 + rr;
#pragma unroll
            for (int n = 0; n < NW; ++n)
#pragma unroll
                for (int t = 0; t < TT; ++t) acc[rr][n][t] = warp_sum(acc[rr][n][t]);
            if (row < p.n_out) {
#pragma unroll
                for (int t = 0; t < TT; ++t) {
                    if (lane == t && t < p.T) {
                        if (MODE == G_QKV) {
                            p.out[(size_t)t * p.n_out + row] = acc[rr][0][t];
                        } else if (MODE == G_RESID) {
                            float* o = p.out + (size_t)t * p.n_out + row;
                            float base = first_rows ? xres[rr] : *o;
                            if (!first_rows)
                                for (int g = 0; g < p.n_add; ++g) base += p.xadd[((size_t)g * p.T + t) * p.n_out + row];
                            *o = base + acc[rr][0][t];
                        } else if (MODE == G_GATEUP) {
                            const float g = acc[rr][0][t], u = acc[rr][NW - 1][t];
                            const float a = silu_f(g) * u;
                            if (f16_out_of_range(a)) atomicOr(p.status, QW_DEV_RANGE);
                            p.out_h[(size_t)t * p.n_out + row] = __float2half_rn(a);
                        } else {
                            if (p.out) p.out[(size_t)t * p.n_out + row] = acc[rr][0][t];
                            best[t] = u64_max(best[t], argmax_key(acc[rr][0][t], row));
                        }
                    }
                }
            }
        }
        first_rows = false;
    }

    if (MODE == G_LMHEAD) {
        __shared__ unsigned long long sbest[GEMV_WARPS][TT];
#pragma unroll
        for (int t = 0; t < TT; ++t)
            if (lane == t) sbest[warp][t] = best[t];
        __syncthreads();
        if (tid < TT && tid < p.T) {
            unsigned long long b = 0ull;
            for (int w = 0; w < GEMV_WARPS; ++w) b = u64_max(b, sbest[w][tid]);
            atomicMax(p.best + tid, b);
        }
    }
}

namespace {

int g_num_sms = 0;

int num_sms() {
    if (g_num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_num_sms <= 0) g_num_sms = 148;
    }
    return g_num_sms;
}

template <int TT, int MODE, int KC, int RPW, int QB>
cudaError_t gemv_go(const LaunchCtx& c, const GemvP& p, int max_ctas) {
    const size_t smem = (size_t)TT * KC * 256 * sizeof(float);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_gemv<TT, MODE, KC, RPW, QB>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int per_cta = GEMV_WARPS * RPW;
    int grid = (p.n_out + per_cta - 1) / per_cta;
    if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
    return launch_k(c, k_gemv<TT, MODE, KC, RPW, QB>, dim3(grid), dim3(GEMV_WARPS * 32), smem, p);
}

// Rows per warp: a lane holds whole rows (K <= 3072) of RPW rows in registers; 4 rows of
// K=1024 (64 registers) for 1-2 tokens, fewer for more tokens or longer rows, so that the
// narrow long-K matrices (o_proj, down_proj: 1024 rows) still spread over >= 256 CTAs.
template <int MODE, int KC, int QB>
cudaError_t gemv_kc(const LaunchCtx& c, const GemvP& p, int max_ctas) {
    constexpr int NW = (MODE == G_GATEUP) ? 2 : 1;
    constexpr int R12 = (KC >= 8 ? 1 : 4 / NW);
    constexpr int R4 = (KC >= 8 ? 1 : 2 / NW);
    if (p.T <= 1) return gemv_go<1, MODE, KC, R12, QB>(c, p, max_ctas);
    if (p.T <= 2) return gemv_go<2, MODE, KC, R12, QB>(c, p, max_ctas);
    if (p.T <= 4) return gemv_go<4, MODE, KC, R4, QB>(c, p, max_ctas);
    return gemv_go<8, MODE, KC, 1, QB>(c, p, max_ctas);
}

// Quantized weights exist only for the projections of the layers (q|k|v and gate/up over the
// hidden size 1024, o_proj and down_proj over 2048 and 3072 inputs).
template <int MODE, int QB>
cudaError_t gemv_dispatch(const LaunchCtx& c, const GemvP& p, int max_ctas) {
    if (p.T < 1 || p.T > 8) return cudaErrorInvalidValue;
    if constexpr (QB == 16) {
        switch (p.K) {
            case 1024: return gemv_kc<MODE, 4, 16>(c, p, max_ctas);
            case 2048: return gemv_kc<MODE, 8, 16>(c, p, max_ctas);
            case 3072: return gemv_kc<MODE, 12, 16>(c, p, max_ctas);
            case 4096: return gemv_kc<MODE, 16, 16>(c, p, max_ctas);
            default: return cudaErrorInvalidValue;
        }
    } else if constexpr (MODE == G_QKV || MODE == G_GATEUP) {
        return p.K == 1024 ? gemv_kc<MODE, 4, QB>(c, p, max_ctas) : cudaErrorInvalidValue;
    } else if constexpr (MODE == G_RESID) {
        if (p.K == 2048) return gemv_kc<MODE, 8, QB>(c, p, max_ctas);
        if (p.K == 3072) return gemv_kc<MODE, 12, QB>(c, p, max_ctas);
        return cudaErrorInvalidValue;
    } else {
        return cudaErrorInvalidValue;
    }
}

template <int MODE>
cudaError_t gemv_any(const LaunchCtx& c, const GemvP& p, int qbits, int max_ctas) {
    if (qbits == 8) return gemv_dispatch<MODE, 8>(c, p, max_ctas);
    if (qbits == 4) return gemv_dispatch<MODE, 4>(c, p, max_ctas);
    return gemv_dispatch<MODE, 16>(c, p, max_ctas);
}

}  // namespace

cudaError_t launch_gemv_qkv(const LaunchCtx& c, int T, const float* x, const bf16* norm_w, float eps,
                            const bf16* W, int n_out, int K, float* out, const QWeights* qw) {
    GemvP p = {};
    p.x = x; p.norm_w = norm_w; p.eps = eps; p.W = W; p.n_out = n_out; p.K = K; p.T = T; p.out = out;
    if (qw) { p.qw = qw->codes; p.sb = qw->sb; }
    return gemv_any<G_QKV>(c, p, qw ? qw->bits : 16, 0);
}

cudaError_t launch_gemv_gateup(const LaunchCtx& c, int T, const float* x, const bf16* norm_w,
                               float eps, const bf16* Wg, const bf16* Wu, int inter, int K, f16* act,
                               int* status, const QWeights* qg, const QWeights* qu, const float* xadd, int n_add) {
    GemvP p = {};
    p.x = x; p.norm_w = norm_w; p.eps = eps; p.W = Wg; p.W2 = Wu; p.n_out = inter; p.K = K; p.T = T;
    p.out_h = act; p.status = status; p.xadd = xadd; p.n_add = xadd ? n_add : 0;
    if (qg) { p.qw = qg->codes; p.sb = qg->sb; p.qw2 = qu->codes; p.sb2 = qu->sb; }
    return gemv_any<G_GATEUP>(c, p, qg ? qg->bits : 16, 0);
}

cudaError_t launch_gemv_resid(const LaunchCtx& c, int T, const f16* act, const bf16* W, int n_out,
                              int K, float* x, const QWeights* qw, const float* xadd, int n_add) {
    GemvP p = {};
    p.act = act; p.W = W; p.n_out = n_out; p.K = K; p.T = T; p.out = x; p.xadd = xadd; p.n_add = xadd ? n_add : 0;
    if (qw) { p.qw = qw->codes; p.sb = qw->sb; }
    return gemv_any<G_RESID>(c, p, qw ? qw->bits : 16, 0);
}

cudaError_t launch_gemv_lmhead(const LaunchCtx& c, int B, const float* x, const int* rows,
                               const bf16* norm_w, float eps, const bf16* E, int vocab, int K,
                               float* logits, unsigned long long* best, const float* xadd, int n_add) {
    GemvP p = {};
    p.x = x; p.rows = rows; p.norm_w = norm_w; p.eps = eps; p.W = E; p.n_out = vocab; p.K = K;
    p.T = B; p.out = logits; p.best = best; p.xadd = xadd; p.n_add = xadd ? n_add : 0;
    return gemv_dispatch<G_LMHEAD, 16>(c, p, num_sms() * 8);
}

// =======================================================================================
// Finalize: unpack the argmax keys into next ids (lowest index wins ties), clear the keys
// for the next call and advance each sequence's length by its token count (Paso 9).
// =======================================================================================
__global__ void k_finalize(StepDesc sd, unsigned long long* best, int32_t* next_ids, KVView kv) {
    pdl_launch();
    pdl_wait();
    for (int b = threadIdx.x; b < sd.B; b += blockDim.x) {
        const unsigned long long key = best[b];
        next_ids[b] = (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
        best[b] = 0ull;
        kv.len[sd.seq[b]] += sd.start[b + 1] - sd.start[b];
    }
}

cudaError_t launch_finalize(const LaunchCtx& c, const StepDesc& sd, unsigned long long* best,
                            int32_t* next_ids, KVView kv) {
    return launch_k(c, k_finalize, dim3(1), dim3(256), 0, sd, best, next_ids, kv);
}

// =======================================================================================
// QK-norm + RoPE + KV append (Paso 5; Paso 4 for the rotation).
// One warp per (token, head) over the fp32 q|k|v projection row; lane l holds dims
// [4l, 4l+4), so dim i and its rotate-half partner i+64 sit in lanes l and l^16.
//   q, k heads: per-head RMSNorm over head_dim with the shared [head_dim] weight, then the
//               rotation by pos * theta^(-i/64) (cos/sin from the fp32 table).
//   v heads   : copied.
// q is written as fp16 [T][n_heads][128]; k and v go (fp16) to the page slot
// page_table[seq][pos / 16] * 16 + pos % 16 of this layer.
// =======================================================================================
__global__ void __launch_bounds__(256) k_qknorm_rope_append(
    int T, int layer, const float* __restrict__ qkv, const bf16* __restrict__ q_norm,
    const bf16* __restrict__ k_norm, float eps, const float* __restrict__ rope_cos,
    const float* __restrict__ rope_sin, int n_heads, int n_kv, TokView tv, KVView kv,
    f16* __restrict__ q_out, int32_t* dbg_pos, int32_t* dbg_slot,
    int* status) {
    pdl_launch();
    pdl_wait();
    const int NH = n_heads + 2 * n_kv;
    const int w = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int t = w / NH, hh = w % NH;
    if (t < T) {
        const float4 xv = *reinterpret_cast<const float4*>(qkv + ((size_t)t * NH + hh) * 128 + lane * 4);
        float y[4] = {xv.x, xv.y, xv.z, xv.w};
        const int pos = tv.pos[t];
        if (hh < n_heads + n_kv) {
            const bf16* nw = (hh < n_heads) ? q_norm : k_norm;
            const float ss = warp_sum(y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3]);
            const float r = rsqrtf(ss * (1.0f / 128.0f) + eps);
            const uint2 wb = *reinterpret_cast<const uint2*>(nw + lane * 4);
            y[0] *= r * bf_lo(wb.x);
            y[1] *= r * bf_hi(wb.x);
            y[2] *= r * bf_lo(wb.y);
            y[3] *= r * bf_hi(wb.y);
            const int i0 = (lane & 15) * 4;
            const float4 cs = *reinterpret_cast<const float4*>(rope_cos + (size_t)pos * 64 + i0);
            const float4 sn = *reinterpret_cast<const float4*>(rope_sin + (size_t)pos * 64 + i0);
            const float c[4] = {cs.x, cs.y, cs.z, cs.w}, s[4] = {sn.x, sn.y, sn.z, sn.w};
            float o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float pj = __shfl_xor_sync(0xffffffffu, y[j], 16);
                o[j] = (lane < 16) ? (y[j] * c[j] - pj * s[j]) : (pj * s[j] + y[j] * c[j]);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) y[j] = o[j];
        }
        if (f16_out_of_range(y[0]) || f16_out_of_range(y[1]) || f16_out_of_range(y[2]) || f16_out_of_range(y[3]))
            atomicOr(status, QW_DEV_RANGE);
        uint2 packed;
        packed.x = pack_h2(y[0], y[1]);
        packed.y = pack_h2(y[2], y[3]);
        if (hh < n_heads) {
            *reinterpret_cast<uint2*>(q_out + ((size_t)t * n_heads + hh) * 128 + lane * 4) = packed;
        } else {
            const int which = (hh - n_heads) / n_kv;  // 0 = K, 1 = V
            const int g = (hh - n_heads) % n_kv;
            const int seq = tv.seq[t];
            const int pi = pos >> 4;
            const int page = (pi < kv.max_pages_per_seq) ? kv.page_table[(size_t)seq * kv.max_pages_per_seq + pi] : -1;
            if (page < 0 || page >= kv.n_pages) {
                if (lane == 0) atomicOr(status, QW_DEV_BAD_POS);
            } else {
                f16* pool = (which == 0 ? kv.k : kv.v) + (size_t)layer * kv.layer_stride;
                f16* dst = pool + (((size_t)page * n_kv + g) * 16 + (pos & 15)) * 128 + lane * 4;
                *reinterpret_cast<uint2*>(dst) = packed;
                if (dbg_pos && which == 0 && g == 0 && lane == 0) {
                    dbg_pos[t] = pos;
                    dbg_slot[t] = page * 16 + (pos & 15);
                }
            }
        }
    }
}

cudaError_t launch_qknorm_rope_append(const LaunchCtx& c, int T, int layer, const float* qkv,
                                      const bf16* q_norm, const bf16* k_norm, float eps,
                                      const float* rope_cos, const float* rope_sin, int n_heads,
                                      int n_kv, TokView tv, KVView kv, f16* q_out,
                                      int32_t* dbg_pos, int32_t* dbg_slot, int* status) {
    const int warps = T * (n_heads + 2 * n_kv);
    return launch_k(c, k_qknorm_rope_append, dim3((warps + 7) / 8), dim3(256), 0, T, layer, qkv,
                    q_norm, k_norm, eps, rope_cos, rope_sin, n_heads, n_kv, tv, kv, q_out,
                    dbg_pos, dbg_slot, status);
}

// =======================================================================================
// Synthetic KV fill with the counter-based SplitMix64 generator (Steele, Lea, Flood 2014):
// element idx -> z = mix(seed + (idx + 1) * golden); b = (int8)(z >> 56); K = b/64, V = b/128
// (exact in fp16).
// =======================================================================================
__device__ __forceinline__ unsigned long long splitmix64_at(unsigned long long seed,
                                                            unsigned long long idx) {
    unsigned long long z = seed + (idx + 1ull) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__global__ void k_kv_fill(KVView kv, int n_layers, int n_kv, int seq, int n_tokens,
                          unsigned long long seed) {
    // grid: (pages of the sequence, n_layers * 2); block: n_kv * 16 * ... threads loop
    const int pi = blockIdx.x;
    const int layer = blockIdx.y >> 1, which = blockIdx.y & 1;
    const int page = kv.page_table[(size_t)seq * kv.max_pages_per_seq + pi];
    if (page < 0) return;
    f16* pool = (which == 0 ? kv.k : kv.v) + (size_t)layer * kv.layer_stride;
    const float scale = which == 0 ? (1.0f / 64.0f) : (1.0f / 128.0f);
    for (int e = threadIdx.x; e < n_kv * 16 * 128; e += blockDim.x) {
        const int g = e / (16 * 128), o = (e / 128) % 16, d = e % 128;
        const int pos = pi * 16 + o;
        float val = 0.f;
        if (pos < n_tokens) {
            const unsigned long long idx =
                (((((unsigned long long)(layer * 2 + which)) << 22 | (unsigned long long)pos) * n_kv + g) * 128 + d);
            const int8_t b = (int8_t)(splitmix64_at(seed, idx) >> 56);
            val = (float)b * scale;
        }
        pool[(((size_t)page * n_kv + g) * 16 + o) * 128 + d] = __float2half_rn(val);
    }
    (void)n_layers;
}

cudaError_t launch_kv_fill(const LaunchCtx& c, KVView kv, int n_layers, int n_kv, int seq,
                           int n_tokens, unsigned long long seed) {
    const int pages = (n_tokens + 15) / 16;
    if (pages == 0) return cudaSuccess;
    return launch_k(c, k_kv_fill, dim3(pages, n_layers * 2), dim3(256), 0, kv, n_layers, n_kv, seq,
                    n_tokens, seed);
}

// =======================================================================================
// Weight conversion bf16 -> fp16 for the packed copies (done once at load). fp16 carries
// every bf16 value of magnitude in [2^-14, 65504] exactly; smaller magnitudes round to the
// fp16 subnormal grid (absolute error <= 2^-25). Values beyond the fp16 range set
// QW_DEV_RANGE in the status word.
// =======================================================================================
__global__ void k_convert_bf16_f16(const bf16* __restrict__ src, f16* __restrict__ dst, size_t n, int* status) {
    const size_t i0 = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
    const size_t stride = (size_t)gridDim.x * blockDim.x * 8;
    for (size_t i = i0; i < n; i += stride) {
        if (i + 8 <= n) {
            const uint4 w = *reinterpret_cast<const uint4*>(src + i);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
            uint32_t o[4];
            bool bad = false;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float a = bf_lo(ws[j]), b = bf_hi(ws[j]);
                bad |= fabsf(a) > 65504.f || fabsf(b) > 65504.f;
                o[j] = pack_h2(a, b);
            }
            *reinterpret_cast<uint4*>(dst + i) = make_uint4(o[0], o[1], o[2], o[3]);
            if (bad) atomicOr(status, QW_DEV_RANGE);
        } else {
            for (size_t j = i; j < n; ++j) {
                const float a = __bfloat162float(src[j]);
                if (fabsf(a) > 65504.f) atomicOr(status, QW_DEV_RANGE);
                dst[j] = __float2half_rn(a);
            }
        }
    }
}

__global__ void k_check_abs(const bf16* __restrict__ w, size_t n, float limit, int* status) {
    bool big = false;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        big |= !(fabsf(__bfloat162float(w[i])) <= limit);
    if (big) atomicOr(status, QW_DEV_RANGE);
}

cudaError_t launch_check_abs(const LaunchCtx& c, const bf16* w, size_t n, float limit, int* status) {
    if (n == 0) return cudaSuccess;
    return launch_k(c, k_check_abs, dim3((unsigned)std::min<size_t>((n + 255) / 256, 1024)), dim3(256), 0, w, n,
                    limit, status);
}

cudaError_t launch_convert_bf16_f16(const LaunchCtx& c, const bf16* src, f16* dst, size_t n, int* status) {
    if (n == 0) return cudaSuccess;
    size_t blocks = (n / 8 + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    return launch_k(c, k_convert_bf16_f16, dim3((unsigned)blocks), dim3(256), 0, src, dst, n, status);
}

// gate/up interleave for the tensor-core SwiGLU: output row r of block b = r / 128 is gate row
// 64 b + r % 128 for r % 128 < 64, else up row 64 b + r % 128 - 64.
__global__ void k_convert_gateup(const bf16* __restrict__ gate, const bf16* __restrict__ up, f16* __restrict__ dst,
                                 int inter, int K, int* status) {
    const int r = blockIdx.x;  // destination row
    const int b = r >> 7, w = r & 127;
    const bf16* src = (w < 64 ? gate : up) + (size_t)(b * 64 + (w & 63)) * K;
    bool big = false;
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        const float v = __bfloat162float(src[k]);
        big |= fabsf(v) > 65504.f;
        dst[(size_t)r * K + k] = __float2half_rn(v);
    }
    if (big) atomicOr(status, QW_DEV_RANGE);
}

cudaError_t launch_convert_gateup(const LaunchCtx& c, const bf16* gate, const bf16* up, f16* dst, int inter, int K,
                                  int* status) {
    return launch_k(c, k_convert_gateup, dim3(2 * inter), dim3(256), 0, gate, up, dst, inter, K, status);
}

// =======================================================================================
// Weight-only grouped affine quantization ("Lo que omite el script": 4- and 8-bit weights):
// each row of a [rows, K] bf16 matrix is cut into groups of 64 inputs; per group, in fp32,
// scale = (max - min) / (2^bits - 1) and bias = min, both rounded to fp16 (how they are
// stored, as one half2 word: scale low, bias high); code q = clamp(rint((w - bias) / scale),
// 0, 2^bits - 1) (q = 0 where the fp16 scale is 0), with IEEE division. Codes are stored one
// per byte (8 bits) or two per byte, the even input in the low nibble (4 bits). The thread of
// a group also writes the dequantized weights scale * q + bias (fp16) into the tensor-core
// copy of the matrix, at row deq_row(r): r, or r's place among interleaved gate/up rows.
// =======================================================================================
__global__ void k_quantize(const bf16* __restrict__ W, int rows, int K, int nbits, uint8_t* __restrict__ codes,
                           uint32_t* __restrict__ sb, f16* __restrict__ deq, int deq_mode) {
    const int G = K / 64;
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= (long long)rows * G) return;
    const int r = (int)(gid / G), g = (int)(gid % G);
    const bf16* src = W + (size_t)r * K + g * 64;
    float w[64];
    float lo = INFINITY, hi = -INFINITY;
#pragma unroll
    for (int i = 0; i < 64; i += 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + i);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            w[i + 2 * j] = bf_lo(u[j]);
            w[i + 2 * j + 1] = bf_hi(u[j]);
        }
    }
#pragma unroll
    for (int i = 0; i < 64; ++i) {
        lo = fminf(lo, w[i]);
        hi = fmaxf(hi, w[i]);
    }
    const float levels = (float)((1 << nbits) - 1);
    const __half s16 = __float2half_rn(__fdiv_rn(hi - lo, levels));
    const __half b16 = __float2half_rn(lo);
    const float s = __half2float(s16), b = __half2float(b16);
    sb[(size_t)r * G + g] = (uint32_t)__half_as_ushort(s16) | ((uint32_t)__half_as_ushort(b16) << 16);
    int dr = r;
    if (deq_mode == 1) dr = (r / 64) * 128 + r % 64;       // gate row among interleaved gate/up rows
    else if (deq_mode == 2) dr = (r / 64) * 128 + 64 + r % 64;  // up row
    f16* drow = deq + (size_t)dr * K + g * 64;
    uint32_t pack = 0;
#pragma unroll
    for (int i = 0; i < 64; ++i) {
        float q = s == 0.f ? 0.f : rintf(__fdiv_rn(w[i] - b, s));
        q = fminf(fmaxf(q, 0.f), levels);
        const uint32_t qi = (uint32_t)q;
        drow[i] = __float2half_rn(fmaf(s, q, b));
        if (nbits == 8) {
            pack |= qi << (8 * (i & 3));
            if ((i & 3) == 3) {
                *reinterpret_cast<uint32_t*>(codes + (size_t)r * K + g * 64 + i - 3) = pack;
                pack = 0;
            }
        } else {
            pack |= qi << (4 * (i & 7));
            if ((i & 7) == 7) {
                *reinterpret_cast<uint32_t*>(codes + ((size_t)r * K + g * 64 + i - 7) / 2) = pack;
                pack = 0;
            }
        }
    }
}

cudaError_t launch_quantize(cudaStream_t st, const bf16* W, int rows, int K, int nbits, uint8_t* codes, uint32_t* sb,
                            f16* deq, int deq_mode) {
    if (K % 64 || (nbits != 8 && nbits != 4)) return cudaErrorInvalidValue;
    const long long groups = (long long)rows * (K / 64);
    const int threads = 128;
    const unsigned blocks = (unsigned)((groups + threads - 1) / threads);
    k_quantize<<<blocks, threads, 0, st>>>(W, rows, K, nbits, codes, sb, deq, deq_mode);
    return cudaGetLastError();
}
