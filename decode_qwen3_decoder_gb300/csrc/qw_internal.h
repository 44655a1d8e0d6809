// Internal declarations shared by the libqw translation units (host runtime + kernels).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qw.h"

typedef __nv_bfloat16 bf16;
typedef __half f16;

// Device status bits (ORed into the workspace status word; read by qw_sync_status).
enum : int {
    QW_DEV_BAD_TOKEN = 1,
    QW_DEV_TIMEOUT = 2,
    QW_DEV_BAD_POS = 4,
    QW_DEV_RANGE = 8,
};

// Per-call batch description, passed by value to the step-begin kernel.
struct StepDesc {
    int B;                       // sequences in the call
    int T;                       // tokens in the call
    int seq[QW_MAX_BATCH];       // sequence id of batch entry b
    int start[QW_MAX_BATCH + 1]; // token offsets: tokens of entry b are [start[b], start[b+1])
};

// Device view of the paged KV cache.
struct KVView {
    int* len;            // [max_seqs] current length of each sequence
    int* page_table;     // [max_seqs][max_pages_per_seq], -1 = no page
    f16* k;              // [n_layers][n_pages][n_kv][page][head_dim]
    f16* v;
    int max_pages_per_seq;
    int n_pages;
    long long layer_stride; // elements per layer of the K (or V) pool
};

// Per-token bookkeeping written by the step-begin kernel.
struct TokView {
    int* seq;  // [T]
    int* pos;  // [T]
    int* last; // [B] row of each entry's last token
    int* slot; // [T] KV slot row page * 16 + pos % 16 of the token (-1: no page reserved)
};

// ---------------------------------------------------------------------------------------
// Small device helpers
// ---------------------------------------------------------------------------------------
#ifdef __CUDACC__
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf2f(bf16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float h_lo(uint32_t w) {
    return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
}
__device__ __forceinline__ float h_hi(uint32_t w) {
    return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
// A value that an fp16 store would not hold (beyond the largest finite fp16, or NaN).
__device__ __forceinline__ bool f16_out_of_range(float v) { return !(fabsf(v) <= 65504.f); }
// Key that orders like the float value, with the lowest index winning ties under max.
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    uint32_t u = __float_as_uint(v);
    uint32_t k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)k << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}
__device__ __forceinline__ unsigned long long u64_max(unsigned long long a, unsigned long long b) {
    return a > b ? a : b;
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = u64_max(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
// Programmatic dependent launch: wait for the upstream grid's memory / let dependents start.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
#endif

// ---------------------------------------------------------------------------------------
// Launchers (defined in the kernel translation units). All return cudaGetLastError().
// ---------------------------------------------------------------------------------------
struct LaunchCtx {
    cudaStream_t stream;
    bool pdl;     // launch with programmatic stream serialization
    int* counter; // incremented per launch (kernel count bookkeeping)
};

#ifdef __CUDACC__
#include <utility>
// Launch a kernel on c.stream, with programmatic stream serialization when c.pdl is set,
// counting the launch in c.counter.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(const LaunchCtx& c, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     Args&&... args) {
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
// launch_k with thread-block clusters of `cluster` CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_kc(const LaunchCtx& c, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      unsigned cluster, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (c.pdl) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    if (c.counter) ++*c.counter;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
#endif

cudaError_t launch_step_begin(const LaunchCtx& c, const StepDesc& sd, const int32_t* ids,
                              const bf16* embed, int vocab, int hidden, float* x, TokView tv,
                              KVView kv, int* status, float* ss = nullptr, const bf16* w = nullptr,
                              f16* xw = nullptr);
cudaError_t launch_rmsnorm(const LaunchCtx& c, const float* x, const int* rows, int n_rows,
                           int hidden, const bf16* w, float eps, f16* h);
cudaError_t launch_convert_bf16_f16(const LaunchCtx& c, const bf16* src, f16* dst, size_t n, int* status);
// Sets QW_DEV_RANGE when some |w[i]| > limit (i < n).
cudaError_t launch_check_abs(const LaunchCtx& c, const bf16* w, size_t n, float limit, int* status);
// Grouped affine weight codes of one matrix [rows, K]: codes (one per byte at 8 bits, two per
// byte at 4, the even input in the low nibble) and one (scale, bias) half2 word per group of
// 64 inputs, scale in the low half.
struct QWeights {
    const uint8_t* codes;
    const uint32_t* sb;
    int bits;
};
cudaError_t launch_quantize(cudaStream_t st, const bf16* W, int rows, int K, int nbits, uint8_t* codes, uint32_t* sb,
                            f16* deq, int deq_mode);
// GEMV family (T <= 8 token rows); with quantized weights (non-NULL QWeights) the bf16
// pointers are not read.
cudaError_t launch_gemv_qkv(const LaunchCtx& c, int T, const float* x, const bf16* norm_w, float eps,
                            const bf16* W, int n_out, int K, float* out, const QWeights* qw = nullptr);
cudaError_t launch_gemv_gateup(const LaunchCtx& c, int T, const float* x, const bf16* norm_w,
                               float eps, const bf16* Wg, const bf16* Wu, int inter, int K, f16* act,
                               int* status, const QWeights* qg = nullptr, const QWeights* qu = nullptr,
                               const float* xadd = nullptr, int n_add = 0);
// x += W act; with xadd, the residual is x + sum_g xadd[g][t][:] (g < n_add) first.
cudaError_t launch_gemv_resid(const LaunchCtx& c, int T, const f16* act, const bf16* W, int n_out,
                              int K, float* x, const QWeights* qw = nullptr, const float* xadd = nullptr,
                              int n_add = 0);
// xadd / n_add: partial vectors [n_add][B][K] added to the rows of x (in order) before the norm
cudaError_t launch_gemv_lmhead(const LaunchCtx& c, int B, const float* x, const int* rows,
                               const bf16* norm_w, float eps, const bf16* E, int vocab, int K,
                               float* logits, unsigned long long* best, const float* xadd = nullptr,
                               int n_add = 0);
// Final RMSNorm + tied LM head + argmax of ONE row (k_lmhead.cu): the embedding streamed through
// a ring of TMA bulk copies; the same operations, in the same order, as launch_gemv_lmhead.
bool lmhead1_ok(int K, int vocab);
cudaError_t launch_lmhead1(const LaunchCtx& c, const float* x, const int* rows, const bf16* norm_w, float eps,
                           const bf16* E, int vocab, int K, float* logits, unsigned long long* best,
                           const float* xadd, int n_add, int* status, int num_sms, int32_t* next_id = nullptr,
                           int* kv_len = nullptr, int seq = 0, int len_add = 0, unsigned int* done = nullptr);
cudaError_t launch_finalize(const LaunchCtx& c, const StepDesc& sd, unsigned long long* best,
                            int32_t* next_ids, KVView kv);
cudaError_t launch_qknorm_rope_append(const LaunchCtx& c, int T, int layer, const float* qkv,
                                      const bf16* q_norm, const bf16* k_norm, float eps,
                                      const float* rope_cos, const float* rope_sin, int n_heads,
                                      int n_kv, TokView tv, KVView kv, f16* q_out,
                                      int32_t* dbg_pos, int32_t* dbg_slot, int* status);
// Decode mode of the paged attention: QK-norm + RoPE + KV append done inside the kernel.
struct AttnFuse {
    const float* qkv;
    const bf16* q_norm;
    const bf16* k_norm;
    float eps;
    const float* rope_cos;
    const float* rope_sin;
    int32_t* dbg_pos;
    int32_t* dbg_slot;
    int* status;
};
// Decode attention of one token (sequence `seq`) over a cache of at most attn_oproj_max_keys()
// keys, fused with o_proj split by KV head: CTA (rb, g) computes the attention of KV head g
// (both its query heads; QK-norm, RoPE; the CTAs with rb == 0 append the new K/V) and the
// o_proj partial of rows [rb * 32, rb * 32 + 32) over that head's 256 inputs into
// part[g][row]; the partials are added to x by the following gate/up and down_proj kernels.
int attn_oproj_max_keys();
cudaError_t launch_attn_oproj(const LaunchCtx& c, int seq, int layer, const AttnFuse& fz, int n_heads, int n_kv,
                              TokView tv, KVView kv, const bf16* Wo, int D, float* part, f16* dbg_attn);
// Batch-1 decode layer as two cluster launches (k_dec1.cu), for hidden 1024, inter
// 128 x {16, 24, 32}, n_kv <= 8 and caches of at most dec1_max_keys() keys.
// Attention kernel: x = xin + sum_{c < n_add} dpart[c]; RMSNorm; q|k|v of KV head g gathered
// in cluster g; QK-norm, RoPE, KV append, attention; o_proj rows of the head's inputs into
// opart[g][D]. Cluster 0 writes x to xout.
struct Dec1Attn {
    const float* xin;
    const float* dpart;  // [n_add][D]
    int n_add;
    float* dclear;       // [dec1_parts()][D] set to zero: the set this layer's MLP kernel adds into
    float* xout;         // [D]
    const bf16* w_in;
    float eps;
    const bf16* Wqkv;    // [QD + 2 KD][D] of the layer
    const bf16* q_norm;
    const bf16* k_norm;
    const float* rope_cos;
    const float* rope_sin;
    KVView kv;
    int layer;
    int seq;             // the token's sequence
    const int* pos;      // [1] its position (written by the step-begin kernel)
    const bf16* Wo;      // [D][QD] of the layer
    float* opart;        // [n_kv][D]
    f16* dbg_attn;       // optional [QD]
    int32_t* dbg_pos;
    int32_t* dbg_slot;
    int* status;
    int n_kv, QD, KD;
    float scale_log2;
    // optional %globaltimer records: CTA c of this launch writes 8 values at
    // trace[((2 layer) * 128 + c) * 8]
    unsigned long long* trace;
};
// MLP kernel: x = xin + sum_{g < n_add} opart[g]; RMSNorm; gate/up + SwiGLU of 16 x 8 CTAs'
// unit slices; split-K down_proj reduced per cluster and added into dpart[c / 2][D]
// (dec1_parts() slots, zero on entry).
// Cluster 0 writes x to xout.
struct Dec1Mlp {
    const float* xin;
    const float* opart;  // [n_add][D]
    int n_add;
    float* xout;         // [D]
    const bf16* w_post;
    float eps;
    const bf16* Wg;      // [I][D] of the layer
    const bf16* Wu;      // [I][D]
    const bf16* WdT;     // [I][D]: down_proj transposed
    float* dpart;        // [dec1_parts()][D], zero on entry: clusters 2k, 2k + 1 add into slot k
    int I;
    int* status;
    int layer;
    unsigned long long* trace;  // as Dec1Attn's, at trace[((2 layer + 1) * 128 + c) * 8]
};
bool dec1_available(int D, int I, int QD, int n_heads, int n_kv);
int dec1_max_keys();
int dec1_parts();
cudaError_t launch_dec1_attn(const LaunchCtx& c, const Dec1Attn& p);
cudaError_t launch_dec1_mlp(const LaunchCtx& c, const Dec1Mlp& p);
// out[i] = x[i] + sum_{c < n} part[c][i], i < D
cudaError_t launch_dec1_sum(const LaunchCtx& c, const float* x, const float* part, int n, int D, float* out);
// dst[z] = src[z] transposed ([rows][cols] -> [cols][rows]), z < batch
cudaError_t launch_transpose_bf16(cudaStream_t st, const bf16* src, int rows, int cols, int batch, bf16* dst);
cudaError_t launch_attn_paged(const LaunchCtx& c, int T, int layer, const f16* q, int n_heads,
                              int n_kv, TokView tv, KVView kv, int chunk, int n_splits,
                              float* part_o, float* part_ml, int* counters, f16* out,
                              const AttnFuse* fuse, const int* decode_seqs);  // host ids (decode) or NULL
// Decode attention split evenly over (token, KV head, page) items for long or many caches;
// q (fp16, normalised and rotated) and the new K/V must already be in place. seqs: host ids
// of the T tokens' sequences; max_keys bounds every cached length + 1.
// tmK / tmV: the K and V pools as [n_layers * n_pages * n_kv * 16, 128] fp16 maps (box 64 x 16,
// 128-byte swizzle).
cudaError_t launch_attn_decode(const LaunchCtx& c, int T, int layer, const f16* q, int n_heads, int n_kv, KVView kv,
                               const CUtensorMap* tmK, const CUtensorMap* tmV, const int* seqs, int max_keys,
                               int max_slots, float* part_o, float* part_ml, int* counters, f16* out, int* status,
                               int num_sms);
// Causal flash attention of a prefill (sequences start empty) over the K/V just appended to
// the paged cache.
// Causal flash attention of a prefill on tcgen05 (S and O in TMEM), K/V from the cache pages
// through the pools' tensor maps.
cudaError_t launch_attn_prefill_tc(const LaunchCtx& c, const StepDesc& sd, const int* tok_pos, int layer, const f16* q,
                                   KVView kv, const CUtensorMap* tmK, const CUtensorMap* tmV, int n_heads, int n_kv,
                                   f16* out, int* status);
// bf16 gate/up [inter][K] -> fp16 rows interleaved per 64: [gate 64b..64b+63][up 64b..64b+63]...
cudaError_t launch_convert_gateup(const LaunchCtx& c, const bf16* gate, const bf16* up, f16* dst, int inter,
                                  int K, int* status);
cudaError_t launch_kv_fill(const LaunchCtx& c, KVView kv, int n_layers, int n_kv, int seq,
                           int n_tokens, unsigned long long seed);

// What the LM head needs from a model (read-only view for entry points in other files).
struct LmHeadView {
    const bf16* final_norm;
    const bf16* embed;
    float eps;
    int vocab;
    int hidden;
};
bool qw_model_lmhead_view(const qw_model* m, LmHeadView* v);
// Records `fmt` as the calling thread's last error and returns s.
qw_status qw_fail(qw_status s, const char* fmt, ...);

// tcgen05 GEMM (T > 8 token rows). Epilogue kinds:
enum GemmEpi : int { EPI_QKV_HEADS = 0, EPI_RESID_F32 = 1, EPI_SILU_MUL = 2, EPI_ARGMAX = 3 };
struct GemmArgs {
    const CUtensorMap* tmA;   // weights [rows_total, K] fp16, box 128 x 64
    const CUtensorMap* tmB;   // activations [T_cap, K] fp16: three maps, boxes of 64/128/256 rows
    int a_row0;               // first weight row of this matrix (layer offset)
    int b_row0;               // first activation row (token offset of the tmB maps)
    int M;                    // weight rows (multiple of 128)
    int K;                    // reduction length (multiple of 64)
    int T;                    // token rows (columns of the transposed product)
    float* out_f32;           // EPI_RESID_F32: x[t][m] (read and written)
    int ld_out;
    f16* out_h;               // EPI_SILU_MUL: act[t][m] (rows interleaved 64 gate / 64 up per tile)
    float* logits;            // EPI_ARGMAX: optional logits[t][m]
    unsigned long long* best; // EPI_ARGMAX: per-token packed argmax keys
    int* status;
    // EPI_QKV_HEADS: per-head QK-norm + RoPE, q out, k/v appended to the paged cache
    f16* q_out;               // [T][n_heads][128]
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
    int num_sms;
};
int sample_max_vocab();  // largest vocabulary qw_sample_top_p takes (8 slices in shared memory)
cudaError_t launch_sample_top_p(cudaStream_t st, int B, int V, const float* logits, size_t ld, float inv_t,
                                unsigned long long tp_fix, const float* uniform, int32_t* next);
cudaError_t launch_gemm_tc(const LaunchCtx& c, int epi, const GemmArgs& a);
bool gemm_tc_encode_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                        uint32_t box_rows);

// Batched decode step as one cooperative kernel (k_step.cu): every layer of a decode step of
// 16-64 sequences. The batch runs as two halves of at most 32 tokens; CTAs [0, gp) compute the
// projections (tcgen05, weights streamed ahead through a TMA ring), CTAs [gp, grid) the
// attention; phases are ordered by counters in global memory.
constexpr int kStepMaxHalf = 32;     // tokens per half
constexpr int kStepDoneSlots = 48;   // completion counters per (layer, half)
constexpr int kStepDoneStride = 32;  // ints between counters (one 128-byte line each)
struct StepKParams {
    int L, D, I, QD, QKVR, n_heads, n_kv;
    float eps, scale_log2;
    const bf16* norms;  // per layer [input D][post-attention D][q_norm 128][k_norm 128]
    const float* rope_cos;
    const float* rope_sin;
    float* x;           // [T][D] residual stream
    f16* q;             // [T][QD] normalised, rotated queries
    f16* attn;          // [T][QD] attention output
    f16* act;           // [T][I] SiLU(gate) * up
    float* part;        // split-K partials [2][units][32][128]
    float* ss;          // [T][D / 128] sums of squares of x per 128-feature block
    f16* xw;            // [2 * kStepMaxHalf][D] fp16(x * w), w = the next RMSNorm's weight
    int* tick;          // [2][tiles] split-K arrival tickets (reset by the last arrival)
    int* done;          // [L][2][kStepDoneSlots][kStepDoneStride] completion counters (zeroed before the launch)
    float* att_po;      // attention partials [T][n_heads][att_stride][128]
    float* att_pml;     // [T][n_heads][att_stride][2]
    int* att_cnt;       // [T][n_kv] split arrival tickets (reset by the last arrival)
    int att_stride;
    TokView tv;
    KVView kv;
    int* status;
    int* abort_g;       // set on a failed wait: every CTA stops
    int T, nh[2], t0[2];
    int chunk, nsplit;  // attention keys per split (multiple of 16), splits per token
    int gp;             // CTAs of the projection role
    float* dbg_hidden;  // optional [L][T][D]
    int32_t* dbg_pos;
    int32_t* dbg_slot;
    f16* dbg_attn;      // optional [L][T][QD]
    unsigned long long wait_ns;  // bound of every wait on another CTA
    int extra;          // extra arrivals the first o_proj unit waits for (0 in normal use)
    unsigned long long* trace;   // optional: per CTA trace_n records of 5 words (see qw_trace_set)
    int trace_n;
};
size_t step_part_floats(int D, int I, int QKVR, int n_kv);
int step_tiles(int D, int I, int QKVR);
bool step_shape_ok(int D, int I, int QD, int QKVR, int n_heads, int n_kv);
int step_smem_bytes();
int step_blocks_per_sm();  // 0: the kernel cannot be resident (no launch possible)
// Tensor maps: weights (q|k|v, o, gate/up, down; boxes of 128 rows) and token operands (xw,
// attn, act; boxes of 32 rows), all fp16 with 64-column boxes and the 128-byte swizzle.
struct StepMaps {
    CUtensorMap w[4];
    CUtensorMap xw, attn, act;
};
cudaError_t launch_decode_step(cudaStream_t st, const StepKParams& p, const StepMaps& maps, int grid);

