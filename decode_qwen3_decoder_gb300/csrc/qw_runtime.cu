// Host runtime of libqw: the C ABI of include/qw.h.
//
// Holds the model configuration, packs the weights into the caller's workspace, builds
// the RoPE table, runs the paged KV allocator, orchestrates the kernels of one prefill or
// decode step, and captures decode steps into CUDA graphs. Everything here is host code;
// all arithmetic of the forward pass runs in the kernels of k_*.cu.
//
// Page: "Dentro de un LLM: Inferencia en Python puro para Qwen3-0.6B en MLX".
#include <algorithm>
#include <array>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <set>
#include <string>
#include <vector>

#include "qw_internal.h"

// ---------------------------------------------------------------------------------------
// Errors
// ---------------------------------------------------------------------------------------
static thread_local std::string g_err;

static qw_status fail(qw_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return s;
}

#define CUDA_TRY(expr)                                                                        \
    do {                                                                                      \
        cudaError_t _e = (expr);                                                              \
        if (_e != cudaSuccess)                                                                \
            return fail(QW_ERR_CUDA, "%s failed: %s (%s:%d)", #expr, cudaGetErrorString(_e), \
                        __FILE__, __LINE__);                                                  \
    } while (0)

#define QW_TRY(expr)                   \
    do {                               \
        qw_status _s = (expr);         \
        if (_s != QW_OK) return _s;    \
    } while (0)

extern "C" const char* qw_last_error(void) { return g_err.c_str(); }

// ---------------------------------------------------------------------------------------
// Configuration and workspace layout
// ---------------------------------------------------------------------------------------
static constexpr int kMaxSplits = 128;   // split-KV partial slots per (token, head)
static constexpr int kSmallT = 8;        // token rows handled by the GEMV family
static constexpr int kLmGemmMinRows = 4; // LM head rows from which the tensor-core GEMM runs
static constexpr long long kLongDecodeKeys = 16384;  // tokens x keys from which decode attention splits evenly
static constexpr int kShortCacheKeys = 4096;  // batched decode: longest cache served by the per-pair kernel

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static bool config_ok(const qw_config* c, std::string* why) {
    auto bad = [&](const char* m) {
        if (why) *why = m;
        return false;
    };
    if (!c) return bad("config is NULL");
    if (c->n_layers < 1) return bad("n_layers must be >= 1");
    if (c->head_dim != 128) return bad("head_dim must be 128");
    if (c->n_kv_heads < 1 || c->n_heads != 2 * c->n_kv_heads) return bad("need n_heads == 2 * n_kv_heads");
    if (c->hidden <= 0 || c->hidden % 256) return bad("hidden must be a positive multiple of 256");
    if (c->inter <= 0 || c->inter % 256) return bad("inter must be a positive multiple of 256");
    if ((c->n_heads * c->head_dim) % 256) return bad("n_heads * head_dim must be a multiple of 256");
    if (c->hidden > 4096 || c->inter > 4096 || c->n_heads * c->head_dim > 4096)
        return bad("GEMV rows are limited to 4096 columns");
    if (c->vocab <= 0 || c->vocab % 128) return bad("vocab must be a positive multiple of 128");
    if (c->page_size != 16) return bad("page_size must be 16");
    if (c->tie_embed != 1) return bad("only the tied LM head is supported");
    if (!(c->rms_eps > 0.f)) return bad("rms_eps must be > 0");
    if (!(c->rope_theta > 1.0)) return bad("rope_theta must be > 1");
    if (c->max_tokens < 1 || c->max_tokens > (1 << 20)) return bad("max_tokens out of range");
    if (c->max_batch < 1 || c->max_batch > QW_MAX_BATCH) return bad("max_batch out of range");
    if (c->max_context < 1 || c->max_context > (1 << 22)) return bad("max_context out of range");
    return true;
}

// The batch-1 decode layer as two cluster kernels: shapes it serves (the device check is
// dec1_available, at init).
static bool dec1_shape(const qw_config& c) {
    return c.hidden == 1024 && c.n_kv_heads <= 8 && (c.inter == 2048 || c.inter == 3072 || c.inter == 4096);
}

struct WsLayout {
    size_t wqkv, wo, wgu, wd, embed16, bqkv, bo, bg, bu, bd, norms, fnorm, rcos, rsin;
    size_t x, h, qkv, q, attn, act, part_o, part_ml, counters;
    size_t tok_seq, tok_pos, tok_slot, last, best, status, gen_tok, gen_out;
    size_t st_part, st_ss, st_xw, st_done, st_tick, st_abort;  // batched decode-step kernel
    size_t op_part;  // o_proj partials of the fused small-batch decode attention [n_kv][4][D]
    size_t bdT, d1_y, d1_dpart;  // batch-1 cluster path: down_proj transposed, layer input x, partials
    size_t total;
    int part_T;
};

static WsLayout layout_for(const qw_config& c) {
    WsLayout L = {};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    const size_t D = c.hidden, I = c.inter, QD = (size_t)c.n_heads * c.head_dim;
    const size_t KD = (size_t)c.n_kv_heads * c.head_dim, NL = c.n_layers;
    const size_t QKV = QD + 2 * KD;
    const size_t T = c.max_tokens;
    L.wqkv = take(NL * QKV * D * 2);
    L.wo = take(NL * D * QD * 2);
    L.wgu = take(NL * 2 * I * D * 2);
    L.wd = take(NL * D * I * 2);
    L.embed16 = take((size_t)c.vocab * D * 2);
    L.bqkv = take(NL * QKV * D * 2);
    L.bo = take(NL * D * QD * 2);
    L.bg = take(NL * I * D * 2);
    L.bu = take(NL * I * D * 2);
    L.bd = take(NL * D * I * 2);
    L.norms = take(NL * (2 * D + 2 * c.head_dim) * 2);
    L.fnorm = take(D * 2);
    L.rcos = take((size_t)c.max_context * 64 * 4);
    L.rsin = take((size_t)c.max_context * 64 * 4);
    L.x = take(T * D * 4);
    L.h = take(std::max(T, (size_t)c.max_batch) * D * 2);
    L.qkv = take(std::min<size_t>(T, kSmallT) * QKV * 4);  // fp32 q|k|v of the small-batch path
    L.q = take(T * QD * 2);
    L.attn = take(T * QD * 2);
    L.act = take(T * I * 2);
    L.part_T = std::min<int>(c.max_tokens, std::max(c.max_batch, kSmallT));
    L.part_o = take((size_t)L.part_T * c.n_heads * kMaxSplits * 128 * 4);
    L.part_ml = take((size_t)L.part_T * c.n_heads * kMaxSplits * 2 * 4);
    L.counters = take((size_t)L.part_T * c.n_kv_heads * 4);
    L.tok_seq = take(T * 4);
    L.tok_pos = take(T * 4);
    L.tok_slot = take(T * 4);
    L.last = take((size_t)c.max_batch * 4);
    L.best = take((size_t)(c.max_batch + 1) * 8);  // argmax keys, then the head's finish counter
    L.status = take(4);
    {
        // batched decode-step kernel: split-K partials, per-block sums of squares of x,
        // completion counters and arrival tickets (adjacent: one memset clears both), abort word
        const int QKVR = (int)QKV;
        L.st_part = take(step_part_floats((int)D, (int)I, QKVR, c.n_kv_heads) * 4);
        L.st_ss = take((size_t)2 * kStepMaxHalf * (D / 128) * 4);
        L.st_xw = take((size_t)2 * kStepMaxHalf * D * 2);
        L.st_done = take((size_t)c.n_layers * 2 * kStepDoneSlots * kStepDoneStride * 4);
        L.st_tick = take((size_t)2 * step_tiles((int)D, (int)I, QKVR) * 4);
        L.st_abort = take(4);
    }
    L.op_part = take((size_t)c.n_kv_heads * 4 * D * 4);
    if (dec1_shape(c)) {
        L.bdT = take(NL * I * D * 2);
        L.d1_y = take(D * 4);
        L.d1_dpart = take((size_t)2 * dec1_parts() * D * 4);  // two sets, alternating by layer
    }
    L.gen_tok = take(T * 4);
    L.gen_out = take((size_t)c.max_batch * ((size_t)c.max_context + 1) * 4);
    L.total = off;
    return L;
}

// ---------------------------------------------------------------------------------------
// Model and KV objects
// ---------------------------------------------------------------------------------------
struct GraphEntry {
    cudaGraphExec_t exec;
    int launches;
    unsigned long long last_use;
};

struct qw_model {
    qw_config cfg;
    WsLayout L;
    char* ws;
    int qkv_rows;
    f16 *wqkv, *wo, *wgu, *wd, *embed16;  // fp16 copies of the bf16 weights (tensor cores)
    bf16 *bqkv, *bo, *bg, *bu, *bd;           // bf16 packed copies (small-batch decode paths)
    bf16 *norms, *fnorm;
    const bf16* embed;
    float *rcos, *rsin, *x, *qkv, *part_o, *part_ml;
    f16 *h, *q, *attn, *act;
    int *counters, *tok_seq, *tok_pos, *tok_slot, *last, *status;
    // batched decode-step kernel (decode steps of 16 .. 2 * kStepMaxHalf tokens)
    bool step_ok;      // shape supported and one CTA per SM can be resident
    bool use_step;     // QW_OPT_DECODE_STEP_KERNEL
    int step_gp;       // CTAs of its projection role
    unsigned long long step_wait_ns;  // bound of its waits on other CTAs
    int step_extra;    // test-only: extra arrivals its first o_proj unit waits for
    float *st_part, *st_ss;
    float* op_part;
    bf16* bdT;          // [n_layers][inter][hidden]: down_proj transposed (batch-1 cluster path)
    float *d1_y, *d1_dpart;
    bool dec1_ok;       // the batch-1 cluster path fits this shape and device
    bool use_dec1;      // QW_OPT_BATCH1_CLUSTERS
    f16* st_xw;
    int *st_done, *st_tick, *st_abort;
    StepMaps st_maps;
    unsigned long long* best;
    unsigned int* lm_done;  // finished-CTA count of the batch-1 LM head (zero between launches)
    int32_t *gen_tok, *gen_out;
    float* dbg_hidden;
    int32_t *dbg_pos, *dbg_slot;
    f16* dbg_attn;
    cudaStream_t cap_stream;
    cudaStream_t aux_stream;   // second half of a split decode batch
    cudaEvent_t ev_fork, ev_join;
    bool split_decode;         // decode batches of >= 16 run as two overlapping halves
    std::map<std::vector<long long>, GraphEntry> graphs;
    // 16: the small-batch GEMVs read the bf16 weights; 8 / 4: they read grouped affine codes of
    // the layers' projections (per layer: q|k|v, o, gate, up, down), whose dequantized values
    // also replaced the tensor-core fp16 copies
    int qbits = 16;
    std::vector<std::array<QWeights, 5>> qlay;
    unsigned long long use_clock;
    int last_launches;
    int num_sms;
    bool pdl;
    bool chain_step;    // set while a multi-step graph captures its second and later steps
    // profiling: events around launches of one kernel kind
    int prof_kind;
    unsigned long long* trace;
    int trace_n;
    std::vector<cudaEvent_t> prof_events;
    unsigned long long prof_gen;
    // TMA descriptors of the tensor-core GEMM operands
    CUtensorMap tm_wqkv, tm_wo, tm_wgu, tm_wd, tm_embed;
    CUtensorMap tm_h[3], tm_attn[3], tm_act[3];  // token boxes of 64, 128, 256 rows
};

struct qw_kv {
    qw_model* m;
    char* pool;
    int max_seqs, n_pages, maxp;
    int* d_len;
    int* d_pt;
    f16* k;
    f16* v;
    long long layer_stride;
    CUtensorMap tm_k, tm_v;  // K / V pools as [rows, 128] fp16 (box 64 x 16, 128-byte swizzle)
    std::vector<int> len;
    std::vector<std::vector<int>> pt;
    std::set<int> free_pages;

    KVView view() const {
        KVView v_;
        v_.len = d_len;
        v_.page_table = d_pt;
        v_.k = k;
        v_.v = v;
        v_.max_pages_per_seq = maxp;
        v_.n_pages = n_pages;
        v_.layer_stride = layer_stride;
        return v_;
    }
};

// ---------------------------------------------------------------------------------------
// Weights
// ---------------------------------------------------------------------------------------
extern "C" size_t qw_model_workspace_bytes(const qw_config* cfg) {
    if (!config_ok(cfg, nullptr)) return 0;
    return layout_for(*cfg).total;
}

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

extern "C" qw_status qw_init_weights(const qw_config* cfg, const qw_weight_ptrs* w, void* dev_workspace,
                                     size_t ws_bytes, void* stream_, qw_model** out) {
    std::string why;
    if (!out) return fail(QW_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!config_ok(cfg, &why)) return fail(QW_ERR_INVALID_ARG, "invalid config: %s", why.c_str());
    if (!w || !w->embed_tokens || !w->norm || !w->layers) return fail(QW_ERR_INVALID_ARG, "weight pointers missing");
    const WsLayout L = layout_for(*cfg);
    if (!dev_workspace || !aligned(dev_workspace, 256)) return fail(QW_ERR_INVALID_ARG, "workspace NULL or not 256-byte aligned");
    if (ws_bytes < L.total) return fail(QW_ERR_INVALID_ARG, "workspace too small: %zu < %zu", ws_bytes, L.total);
    if (!aligned(w->embed_tokens, 16)) return fail(QW_ERR_INVALID_ARG, "embed_tokens not 16-byte aligned");
    for (int l = 0; l < cfg->n_layers; ++l) {
        const qw_layer_ptrs& lp = w->layers[l];
        const void* ps[11] = {lp.input_layernorm, lp.q_proj, lp.k_proj, lp.v_proj, lp.o_proj, lp.q_norm,
                              lp.k_norm, lp.post_attention_layernorm, lp.gate_proj, lp.up_proj, lp.down_proj};
        for (const void* p : ps)
            if (!p) return fail(QW_ERR_INVALID_ARG, "layer %d has a NULL tensor", l);
    }
    cudaStream_t st = (cudaStream_t)stream_;
    qw_model* m = new qw_model();
    m->cfg = *cfg;
    m->L = L;
    m->ws = (char*)dev_workspace;
    const size_t D = cfg->hidden, I = cfg->inter, d = cfg->head_dim;
    const size_t QD = (size_t)cfg->n_heads * d, KD = (size_t)cfg->n_kv_heads * d;
    m->qkv_rows = (int)(QD + 2 * KD);
    char* b = m->ws;
    m->wqkv = (f16*)(b + L.wqkv);
    m->wo = (f16*)(b + L.wo);
    m->wgu = (f16*)(b + L.wgu);
    m->wd = (f16*)(b + L.wd);
    m->embed16 = (f16*)(b + L.embed16);
    m->bqkv = (bf16*)(b + L.bqkv);
    m->bo = (bf16*)(b + L.bo);
    m->bg = (bf16*)(b + L.bg);
    m->bu = (bf16*)(b + L.bu);
    m->bd = (bf16*)(b + L.bd);
    m->norms = (bf16*)(b + L.norms);
    m->fnorm = (bf16*)(b + L.fnorm);
    m->embed = (const bf16*)w->embed_tokens;
    m->rcos = (float*)(b + L.rcos);
    m->rsin = (float*)(b + L.rsin);
    m->x = (float*)(b + L.x);
    m->h = (f16*)(b + L.h);
    m->qkv = (float*)(b + L.qkv);
    m->q = (f16*)(b + L.q);
    m->attn = (f16*)(b + L.attn);
    m->act = (f16*)(b + L.act);
    m->part_o = (float*)(b + L.part_o);
    m->part_ml = (float*)(b + L.part_ml);
    m->counters = (int*)(b + L.counters);
    m->tok_seq = (int*)(b + L.tok_seq);
    m->tok_pos = (int*)(b + L.tok_pos);
    m->tok_slot = (int*)(b + L.tok_slot);
    m->last = (int*)(b + L.last);
    m->best = (unsigned long long*)(b + L.best);
    m->lm_done = (unsigned int*)(m->best + cfg->max_batch);
    m->status = (int*)(b + L.status);
    m->st_part = (float*)(b + L.st_part);
    m->st_ss = (float*)(b + L.st_ss);
    m->op_part = (float*)(b + L.op_part);
    m->bdT = L.bdT ? (bf16*)(b + L.bdT) : nullptr;
    m->d1_y = L.d1_y ? (float*)(b + L.d1_y) : nullptr;
    m->d1_dpart = L.d1_dpart ? (float*)(b + L.d1_dpart) : nullptr;
    m->st_xw = (f16*)(b + L.st_xw);
    m->st_done = (int*)(b + L.st_done);
    m->st_tick = (int*)(b + L.st_tick);
    m->st_abort = (int*)(b + L.st_abort);
    m->gen_tok = (int32_t*)(b + L.gen_tok);
    m->gen_out = (int32_t*)(b + L.gen_out);
    m->use_clock = 0;
    m->last_launches = 0;
    m->pdl = true;
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (m->num_sms <= 0) m->num_sms = 148;

    auto fail_free = [&](qw_status s) {
        delete m;
        return s;
    };
    auto cp = [&](void* dst, const void* src, size_t bytes) {
        return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st);
    };
    if (cudaMemsetAsync(m->status, 0, 4, st) != cudaSuccess) {
        fail(QW_ERR_CUDA, "status clear failed");
        return fail_free(QW_ERR_CUDA);
    }
    // Pack: the projection matrices become fp16 (the tensor-core operand type; exact for
    // every bf16 magnitude in [2^-14, 65504]); per layer q|k|v rows are concatenated into one
    // [qkv_rows, hidden] matrix; gate and up rows are interleaved in blocks of 64 (64 gate
    // rows, then the same 64 up rows) so one 128-row tile holds both halves of SwiGLU. Norm
    // weights stay bf16, copied as [input D][post-attention D][q_norm d][k_norm d].
    LaunchCtx pc = {st, false, nullptr};
    auto cv = [&](f16* dst, const void* src, size_t n) {
        return launch_convert_bf16_f16(pc, (const bf16*)src, dst, n, m->status);
    };
    for (int l = 0; l < cfg->n_layers; ++l) {
        const qw_layer_ptrs& lp = w->layers[l];
        f16* q0 = m->wqkv + (size_t)l * m->qkv_rows * D;
        cudaError_t e = cudaSuccess;
        if (e == cudaSuccess) e = cv(q0, lp.q_proj, QD * D);
        if (e == cudaSuccess) e = cv(q0 + QD * D, lp.k_proj, KD * D);
        if (e == cudaSuccess) e = cv(q0 + (QD + KD) * D, lp.v_proj, KD * D);
        if (e == cudaSuccess) e = cv(m->wo + (size_t)l * D * QD, lp.o_proj, D * QD);
        if (e == cudaSuccess)
            e = launch_convert_gateup(pc, (const bf16*)lp.gate_proj, (const bf16*)lp.up_proj,
                                      m->wgu + (size_t)l * 2 * I * D, (int)I, (int)D, m->status);
        if (e == cudaSuccess) e = cv(m->wd + (size_t)l * D * I, lp.down_proj, D * I);
        // bf16 packed copies (bit-identical) for the bandwidth-bound small-batch paths
        bf16* b0 = m->bqkv + (size_t)l * m->qkv_rows * D;
        if (e == cudaSuccess) e = cp(b0, lp.q_proj, QD * D * 2);
        if (e == cudaSuccess) e = cp(b0 + QD * D, lp.k_proj, KD * D * 2);
        if (e == cudaSuccess) e = cp(b0 + (QD + KD) * D, lp.v_proj, KD * D * 2);
        if (e == cudaSuccess) e = cp(m->bo + (size_t)l * D * QD, lp.o_proj, D * QD * 2);
        if (e == cudaSuccess) e = cp(m->bg + (size_t)l * I * D, lp.gate_proj, I * D * 2);
        if (e == cudaSuccess) e = cp(m->bu + (size_t)l * I * D, lp.up_proj, I * D * 2);
        if (e == cudaSuccess) e = cp(m->bd + (size_t)l * D * I, lp.down_proj, D * I * 2);
        bf16* nb = m->norms + (size_t)l * (2 * D + 2 * d);
        if (e == cudaSuccess) e = cp(nb, lp.input_layernorm, D * 2);
        if (e == cudaSuccess) e = cp(nb + D, lp.post_attention_layernorm, D * 2);
        if (e == cudaSuccess) e = cp(nb + 2 * D, lp.q_norm, d * 2);
        if (e == cudaSuccess) e = cp(nb + 2 * D + d, lp.k_norm, d * 2);
        if (e != cudaSuccess) {
            fail(QW_ERR_CUDA, "weight packing failed: %s", cudaGetErrorString(e));
            return fail_free(QW_ERR_CUDA);
        }
    }
    if (cp(m->fnorm, w->norm, D * 2) != cudaSuccess ||
        cv(m->embed16, w->embed_tokens, (size_t)cfg->vocab * D) != cudaSuccess) {
        fail(QW_ERR_CUDA, "final norm / embedding copy failed");
        return fail_free(QW_ERR_CUDA);
    }
    // An RMSNorm output over n values has |y_i| <= sqrt(n) * |w_i| (since x_i^2 <= n * mean(x^2)),
    // so norm weights below 65504 / sqrt(n) keep every normalised fp16 operand (h, q, k) finite.
    {
        const float lim_d = 65504.f / std::sqrt((float)D), lim_h = 65504.f / std::sqrt((float)d);
        cudaError_t e = cudaSuccess;
        for (int l = 0; l < cfg->n_layers && e == cudaSuccess; ++l) {
            const bf16* nb = m->norms + (size_t)l * (2 * D + 2 * d);
            e = launch_check_abs(pc, nb, 2 * D, lim_d, m->status);
            if (e == cudaSuccess) e = launch_check_abs(pc, nb + 2 * D, 2 * d, lim_h, m->status);
        }
        if (e == cudaSuccess) e = launch_check_abs(pc, m->fnorm, D, lim_d, m->status);
        if (e != cudaSuccess) {
            fail(QW_ERR_CUDA, "norm weight check failed: %s", cudaGetErrorString(e));
            return fail_free(QW_ERR_CUDA);
        }
    }
    // RoPE table (Paso 4): angle = pos * theta^(-i/64), evaluated in fp64, stored as fp32.
    {
        const size_t n = (size_t)cfg->max_context * 64;
        std::vector<float> c(n), s(n);
        for (int i = 0; i < 64; ++i) {
            const double inv = 1.0 / std::pow(cfg->rope_theta, (double)i / 64.0);
            for (int p = 0; p < cfg->max_context; ++p) {
                const double a = (double)p * inv;
                c[(size_t)p * 64 + i] = (float)std::cos(a);
                s[(size_t)p * 64 + i] = (float)std::sin(a);
            }
        }
        if (cudaMemcpyAsync(m->rcos, c.data(), n * 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
            cudaMemcpyAsync(m->rsin, s.data(), n * 4, cudaMemcpyHostToDevice, st) != cudaSuccess) {
            fail(QW_ERR_CUDA, "RoPE table upload failed");
            return fail_free(QW_ERR_CUDA);
        }
        // pageable sources: keep them alive until the copies are done
        if (cudaStreamSynchronize(st) != cudaSuccess) {
            fail(QW_ERR_CUDA, "stream sync failed");
            return fail_free(QW_ERR_CUDA);
        }
    }
    if (cudaMemsetAsync(m->counters, 0, (size_t)L.part_T * cfg->n_kv_heads * 4, st) != cudaSuccess ||
        cudaMemsetAsync(m->best, 0, (size_t)(cfg->max_batch + 1) * 8, st) != cudaSuccess) {
        fail(QW_ERR_CUDA, "workspace clear failed");
        return fail_free(QW_ERR_CUDA);
    }
    {
        int word = 0;
        if (cudaStreamSynchronize(st) != cudaSuccess ||
            cudaMemcpy(&word, m->status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) {
            fail(QW_ERR_CUDA, "weight conversion failed");
            return fail_free(QW_ERR_CUDA);
        }
        if (word & QW_DEV_RANGE) {
            fail(QW_ERR_INVALID_ARG,
                 "a weight is outside the fp16 range (|w| > 65504), or a norm weight exceeds 65504 / sqrt(n)");
            return fail_free(QW_ERR_INVALID_ARG);
        }
    }
    // Tensor maps for the tcgen05 GEMMs: weights as [rows, K] (box 128 x 64) and the
    // activation operands as [rows, K] (box up to 256 x 64).
    const uint64_t NL = cfg->n_layers, TT = std::max<uint64_t>(cfg->max_tokens, cfg->max_batch);
    bool ok = true;
    ok = ok && gemm_tc_encode_map(&m->tm_wqkv, m->wqkv, NL * m->qkv_rows, D, 128);
    ok = ok && gemm_tc_encode_map(&m->tm_wo, m->wo, NL * D, QD, 128);
    ok = ok && gemm_tc_encode_map(&m->tm_wgu, m->wgu, NL * 2 * I, D, 128);
    ok = ok && gemm_tc_encode_map(&m->tm_wd, m->wd, NL * D, I, 128);
    ok = ok && gemm_tc_encode_map(&m->tm_embed, m->embed16, cfg->vocab, D, 128);
    ok = ok && gemm_tc_encode_map(m->tm_h, m->h, TT, D, 0);
    ok = ok && gemm_tc_encode_map(m->tm_attn, m->attn, cfg->max_tokens, QD, 0);
    ok = ok && gemm_tc_encode_map(m->tm_act, m->act, cfg->max_tokens, I, 0);
    if (!ok) {
        fail(QW_ERR_CUDA, "cuTensorMapEncodeTiled failed");
        return fail_free(QW_ERR_CUDA);
    }
    if (cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&m->aux_stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&m->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&m->ev_join, cudaEventDisableTiming) != cudaSuccess) {
        fail(QW_ERR_CUDA, "stream/event creation failed");
        return fail_free(QW_ERR_CUDA);
    }
    m->split_decode = true;
    m->dbg_hidden = nullptr;
    m->dbg_pos = m->dbg_slot = nullptr;
    m->dbg_attn = nullptr;
    m->prof_kind = QW_PROF_OFF;
    m->prof_gen = 0;
    m->trace = nullptr;
    m->trace_n = 0;
    m->step_ok = step_shape_ok((int)D, (int)I, (int)QD, m->qkv_rows, cfg->n_heads, cfg->n_kv_heads) &&
                 step_blocks_per_sm() >= 1 &&
                 m->num_sms >= 16;
    if (m->step_ok) {
        m->st_maps.w[0] = m->tm_wqkv;
        m->st_maps.w[1] = m->tm_wo;
        m->st_maps.w[2] = m->tm_wgu;
        m->st_maps.w[3] = m->tm_wd;
        m->step_ok = gemm_tc_encode_map(&m->st_maps.xw, m->st_xw, 2 * kStepMaxHalf, D, kStepMaxHalf) &&
                     gemm_tc_encode_map(&m->st_maps.attn, m->attn, cfg->max_tokens, QD, kStepMaxHalf) &&
                     gemm_tc_encode_map(&m->st_maps.act, m->act, cfg->max_tokens, I, kStepMaxHalf);
    }
    m->use_step = false;  // opt in with QW_OPT_DECODE_STEP_KERNEL
    m->dec1_ok = m->bdT && dec1_available((int)D, (int)I, (int)QD, cfg->n_heads, cfg->n_kv_heads);
    if (m->dec1_ok && launch_transpose_bf16(st, m->bd, (int)D, (int)I, cfg->n_layers, m->bdT) != cudaSuccess) {
        fail(QW_ERR_CUDA, "down_proj transpose failed");
        return fail_free(QW_ERR_CUDA);
    }
    // QW_OPT_BATCH1_CLUSTERS: on by default for stacks of layers, where each kernel's weight
    // fetch overlaps the previous kernel (one layer measured faster on the per-phase path)
    m->use_dec1 = m->dec1_ok && cfg->n_layers > 1;
    m->step_gp = std::max(1, std::min(64, m->num_sms / 2));
    m->step_wait_ns = 2000000000ull;
    m->step_extra = 0;
    if (cudaMemsetAsync(b + L.st_done, 0, L.st_abort + 4 - L.st_done, st) != cudaSuccess ||
        cudaMemsetAsync(b + L.st_part, 0, L.st_ss - L.st_part, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        fail(QW_ERR_CUDA, "workspace clear failed");
        return fail_free(QW_ERR_CUDA);
    }
    *out = m;
    return QW_OK;
}

extern "C" void qw_free_model(qw_model* m) {
    if (!m) return;
    for (auto& kv : m->graphs) cudaGraphExecDestroy(kv.second.exec);
    if (m->cap_stream) cudaStreamDestroy(m->cap_stream);
    if (m->aux_stream) cudaStreamDestroy(m->aux_stream);
    if (m->ev_fork) cudaEventDestroy(m->ev_fork);
    if (m->ev_join) cudaEventDestroy(m->ev_join);
    delete m;
}

extern "C" qw_status qw_debug_set(qw_model* m, float* dev_hidden, int32_t* dev_positions, int32_t* dev_slots) {
    if (!m) return fail(QW_ERR_INVALID_ARG, "model is NULL");
    if (dev_hidden && (!dev_positions || !dev_slots)) return fail(QW_ERR_INVALID_ARG, "debug buffers incomplete");
    m->dbg_hidden = dev_hidden;
    m->dbg_pos = dev_hidden ? dev_positions : nullptr;
    m->dbg_slot = dev_hidden ? dev_slots : nullptr;
    return QW_OK;
}

extern "C" qw_status qw_debug_set_attn(qw_model* m, void* dev_attn) {
    if (!m) return fail(QW_ERR_INVALID_ARG, "model is NULL");
    m->dbg_attn = reinterpret_cast<f16*>(dev_attn);
    return QW_OK;
}

extern "C" qw_status qw_sample_top_p(int B, int vocab, const float* dev_logits, size_t ld, float temperature,
                                     float top_p, const float* dev_uniform, int32_t* dev_next_ids, void* stream) {
    if (B < 1 || B > 65535) return fail(QW_ERR_INVALID_ARG, "B out of range");
    if (vocab < 1 || ld < (size_t)vocab) return fail(QW_ERR_INVALID_ARG, "vocab < 1 or ld < vocab");
    if (vocab > sample_max_vocab()) return fail(QW_ERR_INVALID_ARG, "vocab above %d", sample_max_vocab());
    if (!dev_logits || !dev_next_ids) return fail(QW_ERR_INVALID_ARG, "NULL buffer");
    if (!std::isfinite(temperature) || temperature < 0.f) return fail(QW_ERR_INVALID_ARG, "bad temperature");
    if (temperature > 0.f && !dev_uniform) return fail(QW_ERR_INVALID_ARG, "NULL uniforms");
    if (!std::isfinite(top_p) || !(top_p > 0.f) || top_p > 1.f) return fail(QW_ERR_INVALID_ARG, "top_p outside (0, 1]");
    // probabilities are summed as integers of 2^-40 (see k_sample.cu)
    const unsigned long long tp_fix = (unsigned long long)std::llround((double)top_p * 1099511627776.0);
    const float inv_t = temperature > 0.f ? 1.f / temperature : 0.f;
    CUDA_TRY(launch_sample_top_p((cudaStream_t)stream, B, vocab, dev_logits, ld, inv_t, tp_fix, dev_uniform,
                                 dev_next_ids));
    return QW_OK;
}

// ---------------------------------------------------------------------------------------
// Weight-only quantization of the layers' projections
// ---------------------------------------------------------------------------------------
struct QuantMat {
    const bf16* src;
    f16* deq;
    int rows, K, deq_mode;
};

static std::array<QuantMat, 5> quant_mats(const qw_model* m, int l) {
    const qw_config& c = m->cfg;
    const size_t D = c.hidden, I = c.inter, QD = (size_t)c.n_heads * c.head_dim, R = m->qkv_rows;
    return {QuantMat{m->bqkv + l * R * D, m->wqkv + l * R * D, (int)R, (int)D, 0},
            QuantMat{m->bo + l * D * QD, m->wo + l * D * QD, (int)D, (int)QD, 0},
            QuantMat{m->bg + l * I * D, m->wgu + l * 2 * I * D, (int)I, (int)D, 1},
            QuantMat{m->bu + l * I * D, m->wgu + l * 2 * I * D, (int)I, (int)D, 2},
            QuantMat{m->bd + l * D * I, m->wd + l * D * I, (int)D, (int)I, 0}};
}

static size_t quant_bytes(const qw_model* m, int bits, std::vector<std::array<QWeights, 5>>* lay, char* base) {
    size_t off = 0;
    auto take = [&](size_t n) {
        const size_t o = off;
        off = align_up(off + n, 256);
        return o;
    };
    if (lay) lay->assign(m->cfg.n_layers, {});
    for (int l = 0; l < m->cfg.n_layers; ++l) {
        const auto mats = quant_mats(m, l);
        for (int i = 0; i < 5; ++i) {
            const size_t codes = take((size_t)mats[i].rows * mats[i].K * bits / 8);
            const size_t sb = take((size_t)mats[i].rows * (mats[i].K / 64) * 4);
            if (lay) (*lay)[l][i] = QWeights{(const uint8_t*)(base + codes), (const uint32_t*)(base + sb), bits};
        }
    }
    return off;
}

extern "C" size_t qw_quantize_bytes(const qw_model* m, int bits) {
    if (!m || (bits != 8 && bits != 4)) return 0;
    return quant_bytes(m, bits, nullptr, nullptr);
}

extern "C" qw_status qw_quantize_weights(qw_model* m, int bits, void* dev_buf, size_t bytes, void* stream_) {
    if (!m) return fail(QW_ERR_INVALID_ARG, "model is NULL");
    if (bits != 8 && bits != 4) return fail(QW_ERR_INVALID_ARG, "bits must be 8 or 4");
    if (m->qbits != 16) return fail(QW_ERR_BAD_STATE, "the weights are already quantized");
    const qw_config& c = m->cfg;
    const int QD = c.n_heads * c.head_dim;
    if (c.hidden != 1024 || (QD != 2048 && QD != 3072) || (c.inter != 2048 && c.inter != 3072))
        return fail(QW_ERR_UNSUPPORTED, "quantized GEMVs cover hidden 1024 with 2048/3072-wide o_proj and down_proj");
    if (!dev_buf || !aligned(dev_buf, 256)) return fail(QW_ERR_INVALID_ARG, "buffer NULL or not 256-byte aligned");
    std::vector<std::array<QWeights, 5>> lay;
    const size_t need = quant_bytes(m, bits, &lay, (char*)dev_buf);
    if (bytes < need) return fail(QW_ERR_INVALID_ARG, "buffer too small: %zu < %zu", bytes, need);
    cudaStream_t st = (cudaStream_t)stream_;
    for (int l = 0; l < c.n_layers; ++l) {
        const auto mats = quant_mats(m, l);
        for (int i = 0; i < 5; ++i)
            CUDA_TRY(launch_quantize(st, mats[i].src, mats[i].rows, mats[i].K, bits, (uint8_t*)lay[l][i].codes,
                                     (uint32_t*)lay[l][i].sb, mats[i].deq, mats[i].deq_mode));
    }
    for (auto& g : m->graphs) cudaGraphExecDestroy(g.second.exec);  // they launch the bf16 GEMVs
    m->graphs.clear();
    m->qlay = std::move(lay);
    m->qbits = bits;
    return QW_OK;
}

extern "C" int qw_last_launch_count(const qw_model* m) { return m ? m->last_launches : 0; }

extern "C" qw_status qw_trace_set(qw_model* m, unsigned long long* dev_buf, int per_cta) {
    if (!m) return fail(QW_ERR_INVALID_ARG, "model is NULL");
    m->trace = per_cta > 0 ? dev_buf : nullptr;
    m->trace_n = dev_buf ? per_cta : 0;
    ++m->prof_gen;
    return QW_OK;
}


extern "C" qw_status qw_set_option(qw_model* m, int option, int value) {
    if (!m) return fail(QW_ERR_INVALID_ARG, "model is NULL");
    switch (option) {
        case QW_OPT_PDL:
            m->pdl = value != 0;
            return QW_OK;
        case QW_OPT_SPLIT_DECODE:
            m->split_decode = value != 0;
            return QW_OK;
        case QW_OPT_DECODE_STEP_KERNEL:
            if (value && !m->step_ok) return fail(QW_ERR_UNSUPPORTED, "decode-step kernel unavailable for this shape");
            m->use_step = value != 0;
            return QW_OK;
        case QW_OPT_STEP_PROJ_CTAS:
            if (value < 1 || value > m->num_sms - 1) return fail(QW_ERR_INVALID_ARG, "projection CTAs outside [1, SMs)");
            m->step_gp = value;
            return QW_OK;
        case QW_OPT_TEST_WAIT_LIMIT_US:
            if (value < 1) return fail(QW_ERR_INVALID_ARG, "wait limit must be >= 1 us");
            m->step_wait_ns = (unsigned long long)value * 1000ull;
            return QW_OK;
        case QW_OPT_TEST_EXTRA_ARRIVALS:
            if (value < 0) return fail(QW_ERR_INVALID_ARG, "extra arrivals must be >= 0");
            m->step_extra = value;
            return QW_OK;
        case QW_OPT_BATCH1_CLUSTERS:
            if (value && !m->dec1_ok) return fail(QW_ERR_UNSUPPORTED, "batch-1 cluster path unavailable for this shape or device");
            m->use_dec1 = value != 0;
            return QW_OK;
        default:
            return fail(QW_ERR_INVALID_ARG, "unknown option %d", option);
    }
}

bool qw_model_lmhead_view(const qw_model* m, LmHeadView* v) {
    if (!m || !v) return false;
    v->final_norm = m->fnorm;
    v->embed = m->embed;
    v->eps = m->cfg.rms_eps;
    v->vocab = m->cfg.vocab;
    v->hidden = m->cfg.hidden;
    return true;
}

qw_status qw_fail(qw_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return s;
}

extern "C" qw_status qw_profile_set(qw_model* m, int kind, void* const* events, int n_events) {
    if (!m) return fail(QW_ERR_INVALID_ARG, "model is NULL");
    if (kind < QW_PROF_OFF || kind > QW_PROF_STEP) return fail(QW_ERR_INVALID_ARG, "unknown kernel kind %d", kind);
    m->prof_events.clear();
    if (kind == QW_PROF_OFF || !events || n_events < 2) {
        m->prof_kind = QW_PROF_OFF;
        return QW_OK;
    }
    for (int i = 0; i < n_events; ++i) m->prof_events.push_back((cudaEvent_t)events[i]);
    m->prof_kind = kind;
    ++m->prof_gen;
    return QW_OK;
}

// Records the profiling events around one launch of `kind` (j-th of the step).
struct ProfScope {
    qw_model* m;
    cudaStream_t st;
    int idx;
    ProfScope(qw_model* m_, int kind, int* counts, cudaStream_t st_) : m(m_), st(st_), idx(-1) {
        if (m->prof_kind != kind) return;
        const int j = counts[kind]++;
        if (2 * j + 1 < (int)m->prof_events.size()) {
            idx = 2 * j;
            record(m->prof_events[idx]);
        }
    }
    // inside stream capture the records become event-record nodes of the graph
    void record(cudaEvent_t ev) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaStreamIsCapturing(st, &cs);
        if (cs == cudaStreamCaptureStatusActive)
            cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
        else
            cudaEventRecord(ev, st);
    }
    ~ProfScope() {
        if (idx >= 0) record(m->prof_events[idx + 1]);
    }
};

// ---------------------------------------------------------------------------------------
// Paged KV cache
// ---------------------------------------------------------------------------------------
static size_t kv_meta_bytes(const qw_model* m, int max_seqs) {
    const int maxp = (m->cfg.max_context + 15) / 16;
    return align_up((size_t)max_seqs * 4, 256) + align_up((size_t)max_seqs * maxp * 4, 256);
}

static size_t kv_page_bytes(const qw_model* m) {  // K + V, all layers, one page
    return (size_t)m->cfg.n_layers * 2 * m->cfg.n_kv_heads * 16 * m->cfg.head_dim * 2;
}

extern "C" size_t qw_kv_pool_bytes(const qw_model* m, int n_pages, int max_seqs) {
    if (!m || n_pages < 1 || max_seqs < 1) return 0;
    return kv_meta_bytes(m, max_seqs) + kv_page_bytes(m) * (size_t)n_pages;
}

extern "C" qw_status qw_kv_alloc(qw_model* m, void* dev_pool, size_t pool_bytes, int max_seqs, void* stream_,
                                 qw_kv** out) {
    if (!out) return fail(QW_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!m || !dev_pool || !aligned(dev_pool, 256)) return fail(QW_ERR_INVALID_ARG, "model/pool NULL or pool not 256-byte aligned");
    if (max_seqs < 1 || max_seqs > (1 << 20)) return fail(QW_ERR_INVALID_ARG, "max_seqs out of range");
    const size_t meta = kv_meta_bytes(m, max_seqs);
    if (pool_bytes < meta + kv_page_bytes(m)) return fail(QW_ERR_INVALID_ARG, "pool too small for one page");
    const long long n_pages = (long long)((pool_bytes - meta) / kv_page_bytes(m));
    if (n_pages > (1ll << 30)) return fail(QW_ERR_INVALID_ARG, "pool too large");
    cudaStream_t st = (cudaStream_t)stream_;
    qw_kv* kv = new qw_kv();
    kv->m = m;
    kv->pool = (char*)dev_pool;
    kv->max_seqs = max_seqs;
    kv->n_pages = (int)n_pages;
    kv->maxp = (m->cfg.max_context + 15) / 16;
    kv->d_len = (int*)kv->pool;
    kv->d_pt = (int*)(kv->pool + align_up((size_t)max_seqs * 4, 256));
    kv->layer_stride = (long long)n_pages * m->cfg.n_kv_heads * 16 * m->cfg.head_dim;
    kv->k = (f16*)(kv->pool + meta);
    kv->v = kv->k + (size_t)m->cfg.n_layers * kv->layer_stride;
    {
        const unsigned long long rows = (unsigned long long)m->cfg.n_layers * n_pages * m->cfg.n_kv_heads * 16;
        if (rows >= (1ull << 31) || !gemm_tc_encode_map(&kv->tm_k, kv->k, rows, m->cfg.head_dim, 16) ||
            !gemm_tc_encode_map(&kv->tm_v, kv->v, rows, m->cfg.head_dim, 16)) {
            delete kv;
            return fail(QW_ERR_INVALID_ARG, "KV pool too large for tensor-map row coordinates");
        }
    }
    kv->len.assign(max_seqs, 0);
    kv->pt.assign(max_seqs, std::vector<int>());
    for (int i = 0; i < kv->n_pages; ++i) kv->free_pages.insert(i);
    if (cudaMemsetAsync(kv->d_len, 0, (size_t)max_seqs * 4, st) != cudaSuccess ||
        cudaMemsetAsync(kv->d_pt, 0xFF, (size_t)max_seqs * kv->maxp * 4, st) != cudaSuccess) {
        delete kv;
        return fail(QW_ERR_CUDA, "KV metadata clear failed");
    }
    *out = kv;
    return QW_OK;
}

extern "C" void qw_free_kv(qw_kv* kv) { delete kv; }

extern "C" qw_status qw_kv_reserve(qw_kv* kv, int seq, int total_tokens, void* stream_) {
    if (!kv) return fail(QW_ERR_INVALID_ARG, "kv is NULL");
    if (seq < 0 || seq >= kv->max_seqs) return fail(QW_ERR_INVALID_ARG, "seq id %d out of range", seq);
    if (total_tokens < 0 || total_tokens > kv->m->cfg.max_context)
        return fail(QW_ERR_INVALID_ARG, "total_tokens %d outside [0, max_context]", total_tokens);
    std::vector<int>& t = kv->pt[seq];
    const int need = (total_tokens + 15) / 16 - (int)t.size();
    if (need <= 0) return QW_OK;
    if (need > (int)kv->free_pages.size())
        return fail(QW_ERR_KV_FULL, "KV cache full: %d pages needed, %zu free", need, kv->free_pages.size());
    const int old = (int)t.size();
    for (int i = 0; i < need; ++i) {
        t.push_back(*kv->free_pages.begin());
        kv->free_pages.erase(kv->free_pages.begin());
    }
    CUDA_TRY(cudaMemcpyAsync(kv->d_pt + (size_t)seq * kv->maxp + old, t.data() + old, (size_t)need * 4,
                             cudaMemcpyHostToDevice, (cudaStream_t)stream_));
    return QW_OK;
}

extern "C" qw_status qw_kv_reset(qw_kv* kv, int seq, void* stream_) {
    if (!kv) return fail(QW_ERR_INVALID_ARG, "kv is NULL");
    if (seq < -1 || seq >= kv->max_seqs) return fail(QW_ERR_INVALID_ARG, "seq id %d out of range", seq);
    cudaStream_t st = (cudaStream_t)stream_;
    const int a = seq < 0 ? 0 : seq, b = seq < 0 ? kv->max_seqs : seq + 1;
    for (int s = a; s < b; ++s) {
        for (int p : kv->pt[s]) kv->free_pages.insert(p);
        kv->pt[s].clear();
        kv->len[s] = 0;
    }
    CUDA_TRY(cudaMemsetAsync(kv->d_len + a, 0, (size_t)(b - a) * 4, st));
    CUDA_TRY(cudaMemsetAsync(kv->d_pt + (size_t)a * kv->maxp, 0xFF, (size_t)(b - a) * kv->maxp * 4, st));
    return QW_OK;
}

extern "C" qw_status qw_kv_truncate(qw_kv* kv, int seq, int n_tokens, void* stream_) {
    if (!kv) return fail(QW_ERR_INVALID_ARG, "kv is NULL");
    if (seq < 0 || seq >= kv->max_seqs) return fail(QW_ERR_INVALID_ARG, "seq id %d out of range", seq);
    if (n_tokens < 0 || n_tokens > kv->len[seq])
        return fail(QW_ERR_INVALID_ARG, "n_tokens %d outside [0, length %d]", n_tokens, kv->len[seq]);
    const int n = n_tokens;
    CUDA_TRY(cudaMemcpyAsync(kv->d_len + seq, &n, 4, cudaMemcpyHostToDevice, (cudaStream_t)stream_));
    kv->len[seq] = n_tokens;
    return QW_OK;
}

extern "C" int qw_kv_free_pages(const qw_kv* kv) { return kv ? (int)kv->free_pages.size() : -1; }

extern "C" int qw_kv_length(const qw_kv* kv, int seq) {
    if (!kv || seq < 0 || seq >= kv->max_seqs) return -1;
    return kv->len[seq];
}

extern "C" int qw_kv_page_table(const qw_kv* kv, int seq, int32_t* host_out, int max_pages) {
    if (!kv || seq < 0 || seq >= kv->max_seqs) return fail(QW_ERR_INVALID_ARG, "bad kv or seq id");
    const std::vector<int>& t = kv->pt[seq];
    if (host_out)
        for (int i = 0; i < (int)t.size() && i < max_pages; ++i) host_out[i] = t[i];
    return (int)t.size();
}

extern "C" qw_status qw_kv_pool_ptrs(const qw_kv* kv, void** dev_k, void** dev_v, int* n_pages) {
    if (!kv) return fail(QW_ERR_INVALID_ARG, "kv is NULL");
    if (dev_k) *dev_k = kv->k;
    if (dev_v) *dev_v = kv->v;
    if (n_pages) *n_pages = kv->n_pages;
    return QW_OK;
}

extern "C" qw_status qw_kv_fill_synthetic(qw_kv* kv, int seq, int n_tokens, uint64_t seed, void* stream_) {
    if (!kv) return fail(QW_ERR_INVALID_ARG, "kv is NULL");
    if (seq < 0 || seq >= kv->max_seqs) return fail(QW_ERR_INVALID_ARG, "seq id out of range");
    if (n_tokens < 0 || n_tokens > (1 << 22)) return fail(QW_ERR_INVALID_ARG, "n_tokens out of range");
    if (kv->len[seq] != 0) return fail(QW_ERR_BAD_STATE, "sequence %d is not empty", seq);
    if ((int)kv->pt[seq].size() * 16 < n_tokens) return fail(QW_ERR_KV_FULL, "sequence %d reserved for fewer tokens", seq);
    cudaStream_t st = (cudaStream_t)stream_;
    LaunchCtx c = {st, false, nullptr};
    CUDA_TRY(launch_kv_fill(c, kv->view(), kv->m->cfg.n_layers, kv->m->cfg.n_kv_heads, seq, n_tokens, seed));
    const int n = n_tokens;
    CUDA_TRY(cudaMemcpyAsync(kv->d_len + seq, &n, 4, cudaMemcpyHostToDevice, st));
    kv->len[seq] = n_tokens;
    return QW_OK;
}

// ---------------------------------------------------------------------------------------
// One step of the forward pass (prefill or decode)
// ---------------------------------------------------------------------------------------
struct SplitPlan {
    int chunk, n_splits;
};

static SplitPlan plan_splits(const qw_model* m, int T, int max_keys) {
    // aim for ~4 CTAs per SM over T * n_kv (token, KV head) pairs; chunks are whole pages
    const int pairs = T * m->cfg.n_kv_heads;
    int want = (4 * m->num_sms + pairs - 1) / pairs;
    want = std::max(1, std::min(want, kMaxSplits));
    int chunk = (max_keys + want - 1) / want;
    chunk = std::max(64, (chunk + 15) / 16 * 16);
    int n = (max_keys + chunk - 1) / chunk;
    while (n > kMaxSplits) {
        chunk += 16;
        n = (max_keys + chunk - 1) / chunk;
    }
    return {chunk, std::max(n, 1)};
}

// A decode step of one token (bf16 weights, short cache) runs each layer as two cluster
// launches; the LM head then adds the last layer's down_proj partials to x.
static bool dec1_step(const qw_model* m, const StepDesc& sd, bool prefill, int max_keys) {
    return m->use_dec1 && !prefill && sd.T == 1 && m->qbits == 16 && max_keys <= dec1_max_keys();
}

// Token rows [t0, t0 + n) of a step through every layer, on stream st. The rows of a
// decode step are independent sequences, so a batch can run as several such ranges on
// different streams; every buffer is addressed at row t0 (the tensor-core operands through
// the TMA row offset).
static qw_status run_layers(qw_model* m, qw_kv* kv, const StepDesc& sd, bool prefill, int max_keys, int t0, int n,
                            cudaStream_t st, bool dbg, int* launches, int* pc) {
    const qw_config& c = m->cfg;
    const bool pdl_on = m->pdl && m->prof_kind == QW_PROF_OFF;  // events must bracket launches
    LaunchCtx lc = {st, false, launches};  // the first launch of a range follows a full dependency
#define LAUNCH(expr)        \
    do {                    \
        CUDA_TRY(expr);     \
        lc.pdl = pdl_on;    \
    } while (0)
#define PROF(kind) ProfScope prof_scope_(m, kind, pc, st)
    const int T = n;
    const int D = c.hidden, I = c.inter, QD = c.n_heads * c.head_dim, d = c.head_dim;
    const KVView kvv = kv->view();
    const TokView tv = {m->tok_seq + t0, m->tok_pos + t0, m->last, m->tok_slot + t0};
    const bool small = sd.T <= kSmallT;
    const SplitPlan sp = plan_splits(m, T, max_keys);
    // small decode batches over long caches: separate QK-norm/RoPE/append, then the
    // evenly split decode attention (short caches keep the fused per-pair kernel)
    const bool long_decode = !prefill && small && (long long)T * max_keys >= kLongDecodeKeys;
    // decode of one token over a short cache (bf16 weights): attention and o_proj in one kernel,
    // its per-KV-head partials added to x by the gate/up and down_proj kernels
    const bool fuse_ao = !prefill && small && !long_decode && m->qbits == 16 && T == 1 &&
                         max_keys <= attn_oproj_max_keys() && D % 32 == 0;
    const float* xadd = fuse_ao ? m->op_part : nullptr;
    float* x = m->x + (size_t)t0 * D;
    f16* h = m->h + (size_t)t0 * D;
    f16* q = m->q + (size_t)t0 * QD;
    f16* attn = m->attn + (size_t)t0 * QD;
    f16* act = m->act + (size_t)t0 * I;
    float* qkv = m->qkv + (size_t)t0 * m->qkv_rows;
    float* part_o = m->part_o + (size_t)t0 * c.n_heads * kMaxSplits * 128;
    float* part_ml = m->part_ml + (size_t)t0 * c.n_heads * kMaxSplits * 2;
    int* counters = m->counters + (size_t)t0 * c.n_kv_heads;
    int32_t* dbg_pos = dbg ? m->dbg_pos + t0 : nullptr;
    int32_t* dbg_slot = dbg ? m->dbg_slot + t0 : nullptr;
    // SMs a decode GEMM of one half of the two-stream split may spread over: 3/8 of the GPU
    // (32 CTAs for q|k|v, 48 for gate/up, 7-way split-K clusters for o_proj and down_proj at
    // 152 SMs), so that the other half's attention keeps the rest. Measured at B = 64 x 1024
    // keys on one box: 3029 us per step with every GEMM spread over all SMs, 2908 with 1/2,
    // 2760 with 1/3, 2687 with 3/8, 3000 with 1/4.
    const int gsms = (!prefill && T < sd.T) ? std::max(8, m->num_sms * 3 / 8) : m->num_sms;
    if (dec1_step(m, sd, prefill, max_keys)) {
        // x (m->x) -> [attention kernel: x + partials into d1_y, o_proj partials] -> [MLP
        // kernel: d1_y + o_proj partials into m->x, down_proj partials] -> next layer
        const int np = dec1_parts();
        for (int l = 0; l < c.n_layers; ++l) {
            const bf16* nb = m->norms + (size_t)l * (2 * D + 2 * d);
            Dec1Attn a = {};
            // layer l's attention kernel clears set l % 2, its MLP kernel adds into it, and the
            // next layer's attention kernel (or the LM head) reads it
            float* dset = m->d1_dpart + (size_t)(l & 1) * np * D;
            float* dprev = m->d1_dpart + (size_t)((l + 1) & 1) * np * D;
            a.xin = m->x; a.dpart = dprev; a.n_add = l == 0 ? 0 : np; a.dclear = dset; a.xout = m->d1_y;
            a.w_in = nb; a.eps = c.rms_eps; a.Wqkv = m->bqkv + (size_t)l * m->qkv_rows * D;
            a.q_norm = nb + 2 * D; a.k_norm = nb + 2 * D + d; a.rope_cos = m->rcos; a.rope_sin = m->rsin;
            a.kv = kvv; a.layer = l; a.seq = sd.seq[0]; a.pos = tv.pos;
            a.Wo = m->bo + (size_t)l * D * QD; a.opart = m->op_part;
            a.dbg_attn = (dbg && m->dbg_attn) ? m->dbg_attn + (size_t)l * QD : nullptr;
            a.dbg_pos = l == 0 ? dbg_pos : nullptr; a.dbg_slot = l == 0 ? dbg_slot : nullptr;
            a.status = m->status; a.n_kv = c.n_kv_heads; a.QD = QD; a.KD = c.n_kv_heads * d;
            a.scale_log2 = 0.08838834764831845f * 1.4426950408889634f;  // 128^-0.5 * log2(e)
            a.trace = m->trace;
            {
                PROF(QW_PROF_ATTN);
                LAUNCH(launch_dec1_attn(lc, a));
            }
            Dec1Mlp f = {};
            f.xin = m->d1_y; f.opart = m->op_part; f.n_add = c.n_kv_heads; f.xout = m->x;
            f.w_post = nb + D; f.eps = c.rms_eps;
            f.Wg = m->bg + (size_t)l * I * D; f.Wu = m->bu + (size_t)l * I * D; f.WdT = m->bdT + (size_t)l * I * D;
            f.dpart = dset; f.I = I; f.status = m->status; f.layer = l; f.trace = m->trace;
            {
                PROF(QW_PROF_GATEUP);
                LAUNCH(launch_dec1_mlp(lc, f));
            }
            if (dbg) LAUNCH(launch_dec1_sum(lc, m->x, dset, np, D, m->dbg_hidden + (size_t)l * D));
        }
        return QW_OK;
    }
    for (int l = 0; l < c.n_layers; ++l) {
        const bf16* nb = m->norms + (size_t)l * (2 * D + 2 * d);
        const bf16* w_in = nb;
        const bf16* w_post = nb + D;
        const bf16* w_qn = nb + 2 * D;
        const bf16* w_kn = nb + 2 * D + d;
        int32_t* lpos = l == 0 ? dbg_pos : nullptr;
        int32_t* lslot = l == 0 ? dbg_slot : nullptr;
        const QWeights* qq = m->qbits != 16 ? m->qlay[l].data() : nullptr;  // quantized projections
        // --- attention sublayer (Paso 5) ---
        if (small) {
            PROF(QW_PROF_QKV);
            LAUNCH(launch_gemv_qkv(lc, T, x, w_in, c.rms_eps, m->bqkv + (size_t)l * m->qkv_rows * D, m->qkv_rows, D,
                                   qkv, qq ? &qq[0] : nullptr));
        } else {
            {
                PROF(QW_PROF_RMSNORM);
                LAUNCH(launch_rmsnorm(lc, x, nullptr, T, D, w_in, c.rms_eps, h));
            }
            PROF(QW_PROF_QKV);
            // q|k|v projection with the per-head QK-norm, RoPE and the KV append in its epilogue
            GemmArgs g = {};
            g.tmA = &m->tm_wqkv; g.tmB = m->tm_h; g.b_row0 = t0;
            g.a_row0 = l * m->qkv_rows; g.M = m->qkv_rows; g.K = D; g.T = T;
            g.status = m->status; g.num_sms = gsms;
            g.q_out = q; g.q_norm = w_qn; g.k_norm = w_kn; g.eps = c.rms_eps;
            g.rope_cos = m->rcos; g.rope_sin = m->rsin; g.tv = tv; g.kv = kvv; g.layer = l;
            g.n_heads = c.n_heads; g.n_kv = c.n_kv_heads;
            g.dbg_pos = lpos; g.dbg_slot = lslot;
            LAUNCH(launch_gemm_tc(lc, EPI_QKV_HEADS, g));
        }
        if (small) {
            if (prefill) {
                {
                    PROF(QW_PROF_ROPE);
                    LAUNCH(launch_qknorm_rope_append(lc, T, l, qkv, w_qn, w_kn, c.rms_eps, m->rcos, m->rsin,
                                                     c.n_heads, c.n_kv_heads, tv, kvv, q, lpos, lslot, m->status));
                }
                PROF(QW_PROF_ATTN);
                LAUNCH(launch_attn_paged(lc, T, l, q, c.n_heads, c.n_kv_heads, tv, kvv, sp.chunk, sp.n_splits,
                                         part_o, part_ml, counters, attn, nullptr, nullptr));
            } else if (long_decode) {
                {
                    PROF(QW_PROF_ROPE);
                    LAUNCH(launch_qknorm_rope_append(lc, T, l, qkv, w_qn, w_kn, c.rms_eps, m->rcos, m->rsin,
                                                     c.n_heads, c.n_kv_heads, tv, kvv, q, lpos, lslot, m->status));
                }
                PROF(QW_PROF_ATTN);
                LAUNCH(launch_attn_decode(lc, T, l, q, c.n_heads, c.n_kv_heads, kvv, &kv->tm_k, &kv->tm_v, sd.seq + t0,
                                          max_keys, kMaxSplits,
                                          part_o, part_ml, counters, attn, m->status, m->num_sms));
            } else if (fuse_ao) {
                AttnFuse fz = {qkv, w_qn, w_kn, c.rms_eps, m->rcos, m->rsin, lpos, lslot, m->status};
                PROF(QW_PROF_ATTN);
                LAUNCH(launch_attn_oproj(lc, sd.seq[t0], l, fz, c.n_heads, c.n_kv_heads, tv, kvv, m->bo + (size_t)l * D * QD, D,
                                         m->op_part,
                                         (dbg && m->dbg_attn) ? m->dbg_attn + ((size_t)l * sd.T + t0) * QD : nullptr));
            } else {
                // decode: one new token per sequence; QK-norm, RoPE and the KV append run inside
                AttnFuse fz = {qkv, w_qn, w_kn, c.rms_eps, m->rcos, m->rsin, lpos, lslot, m->status};
                PROF(QW_PROF_ATTN);
                LAUNCH(launch_attn_paged(lc, T, l, q, c.n_heads, c.n_kv_heads, tv, kvv, sp.chunk, sp.n_splits,
                                         part_o, part_ml, counters, attn, &fz, sd.seq + t0));
            }
        } else {
            // q, k, v were normalised, rotated and appended by the projection's epilogue
            PROF(QW_PROF_ATTN);
            if (prefill)
                LAUNCH(launch_attn_prefill_tc(lc, sd, m->tok_pos, l, q, kvv, &kv->tm_k, &kv->tm_v, c.n_heads,
                                              c.n_kv_heads, attn, m->status));
            else if (max_keys <= kShortCacheKeys)  // light per-pair kernel: overlaps the other half's GEMMs
                LAUNCH(launch_attn_paged(lc, T, l, q, c.n_heads, c.n_kv_heads, tv, kvv, sp.chunk, sp.n_splits,
                                         part_o, part_ml, counters, attn, nullptr, sd.seq + t0));
            else
                LAUNCH(launch_attn_decode(lc, T, l, q, c.n_heads, c.n_kv_heads, kvv, &kv->tm_k, &kv->tm_v, sd.seq + t0,
                                          max_keys, kMaxSplits,
                                          part_o, part_ml, counters, attn, m->status, m->num_sms));
        }
        if (dbg && m->dbg_attn && !fuse_ao)
            CUDA_TRY(cudaMemcpyAsync(m->dbg_attn + ((size_t)l * sd.T + t0) * QD, attn, (size_t)T * QD * sizeof(f16),
                                     cudaMemcpyDeviceToDevice, st));
        if (fuse_ao) {
            // o_proj ran inside the attention kernel
        } else if (small) {
            PROF(QW_PROF_OPROJ);
            LAUNCH(launch_gemv_resid(lc, T, attn, m->bo + (size_t)l * D * QD, D, QD, x, qq ? &qq[1] : nullptr));
        } else {
            PROF(QW_PROF_OPROJ);
            GemmArgs g = {};
            g.tmA = &m->tm_wo; g.tmB = m->tm_attn; g.b_row0 = t0;
            g.a_row0 = l * D; g.M = D; g.K = QD; g.T = T;
            g.out_f32 = x; g.ld_out = D; g.status = m->status; g.num_sms = gsms;
            LAUNCH(launch_gemm_tc(lc, EPI_RESID_F32, g));
        }
        // --- feed-forward sublayer (Paso 6) ---
        if (small) {
            {
                PROF(QW_PROF_GATEUP);
                LAUNCH(launch_gemv_gateup(lc, T, x, w_post, c.rms_eps, m->bg + (size_t)l * I * D,
                                          m->bu + (size_t)l * I * D, I, D, act, m->status, qq ? &qq[2] : nullptr,
                                          qq ? &qq[3] : nullptr, xadd, c.n_kv_heads));
            }
            PROF(QW_PROF_DOWN);
            LAUNCH(launch_gemv_resid(lc, T, act, m->bd + (size_t)l * D * I, D, I, x, qq ? &qq[4] : nullptr, xadd,
                                     c.n_kv_heads));
        } else {
            {
                PROF(QW_PROF_RMSNORM);
                LAUNCH(launch_rmsnorm(lc, x, nullptr, T, D, w_post, c.rms_eps, h));
            }
            GemmArgs g = {};
            g.tmA = &m->tm_wgu; g.tmB = m->tm_h; g.b_row0 = t0;
            g.a_row0 = l * 2 * I; g.M = 2 * I; g.K = D; g.T = T;
            g.out_h = act; g.ld_out = I; g.status = m->status; g.num_sms = gsms;
            {
                PROF(QW_PROF_GATEUP);
                LAUNCH(launch_gemm_tc(lc, EPI_SILU_MUL, g));
            }
            GemmArgs g2 = {};
            g2.tmA = &m->tm_wd; g2.tmB = m->tm_act; g2.b_row0 = t0;
            g2.a_row0 = l * D; g2.M = D; g2.K = I; g2.T = T;
            g2.out_f32 = x; g2.ld_out = D; g2.status = m->status; g2.num_sms = gsms;
            PROF(QW_PROF_DOWN);
            LAUNCH(launch_gemm_tc(lc, EPI_RESID_F32, g2));
        }
        if (dbg)
            CUDA_TRY(cudaMemcpyAsync(m->dbg_hidden + ((size_t)l * sd.T + t0) * D, x, (size_t)T * D * 4,
                                     cudaMemcpyDeviceToDevice, st));
    }
#undef PROF
#undef LAUNCH
    return QW_OK;
}

static qw_status run_step(qw_model* m, qw_kv* kv, const StepDesc& sd, bool prefill, int max_keys,
                          const int32_t* tokens, float* logits, int32_t* next, cudaStream_t st,
                          bool allow_debug, int* launches) {
    const qw_config& c = m->cfg;
    const int T = sd.T, B = sd.B;
    const int D = c.hidden, I = c.inter, QD = c.n_heads * c.head_dim;
    const KVView kvv = kv->view();
    TokView tv = {m->tok_seq, m->tok_pos, m->last, m->tok_slot};
    const bool dbg = allow_debug && m->dbg_hidden;
    const bool small = T <= kSmallT;
    if (!small && !prefill && T > m->L.part_T) return fail(QW_ERR_UNSUPPORTED, "decode batch beyond partial buffers");

    int pc[16] = {0};
    // The first kernel of a step waits for everything before it, so kernels of this step may
    // read state written by earlier steps before their own wait. Inside a multi-step graph it
    // is launched early (programmatic overlap with the previous step's last kernel) but lets
    // its dependents start only once its own dependency wait has returned.
    const LaunchCtx lc0 = {st, m->chain_step && m->pdl && m->prof_kind == QW_PROF_OFF, launches};
    const bool engine = !prefill && m->use_step && m->qbits == 16 && T >= 16 && T <= 2 * kStepMaxHalf &&
                        (m->prof_kind == QW_PROF_OFF || m->prof_kind == QW_PROF_STEP);
    CUDA_TRY(launch_step_begin(lc0, sd, tokens, m->embed, c.vocab, D, m->x, tv, kvv, m->status,
                               engine ? m->st_ss : nullptr, m->norms, m->st_xw));
    if (engine) {
        // every layer of the step in one cooperative kernel (counters cleared first)
        CUDA_TRY(cudaMemsetAsync(m->st_done, 0, (size_t)c.n_layers * 2 * kStepDoneSlots * kStepDoneStride * 4, st));
        StepKParams sp = {};
        sp.L = c.n_layers; sp.D = D; sp.I = I; sp.QD = QD; sp.QKVR = m->qkv_rows;
        sp.n_heads = c.n_heads; sp.n_kv = c.n_kv_heads; sp.eps = c.rms_eps;
        sp.scale_log2 = 0.08838834764831845f * 1.4426950408889634f;  // 128^-0.5 * log2(e)
        sp.norms = m->norms; sp.rope_cos = m->rcos; sp.rope_sin = m->rsin;
        sp.x = m->x; sp.q = m->q; sp.attn = m->attn; sp.act = m->act;
        sp.part = m->st_part; sp.ss = m->st_ss; sp.xw = m->st_xw; sp.tick = m->st_tick; sp.done = m->st_done;
        sp.att_po = m->part_o; sp.att_pml = m->part_ml; sp.att_cnt = m->counters; sp.att_stride = kMaxSplits;
        sp.tv = tv; sp.kv = kvv; sp.status = m->status; sp.abort_g = m->st_abort;
        sp.T = T;
        sp.nh[0] = T / 2; sp.nh[1] = T - T / 2;
        sp.t0[0] = 0; sp.t0[1] = T / 2;
        sp.gp = m->step_gp;
        {
            // attention units: ~3 per attention warp per layer and half
            const int pairs = sp.nh[1] * c.n_kv_heads;
            const int warps = (m->num_sms - sp.gp) * 8;
            const int want = std::max(1, std::min(kMaxSplits, (3 * warps + pairs - 1) / pairs));
            int chunk = std::max(64, ((max_keys + want - 1) / want + 15) / 16 * 16);
            while ((max_keys + chunk - 1) / chunk > kMaxSplits) chunk += 16;
            sp.chunk = chunk;
            sp.nsplit = (max_keys + chunk - 1) / chunk;
        }
        sp.dbg_hidden = dbg ? m->dbg_hidden : nullptr;
        sp.dbg_pos = dbg ? m->dbg_pos : nullptr;
        sp.dbg_slot = dbg ? m->dbg_slot : nullptr;
        sp.dbg_attn = dbg ? m->dbg_attn : nullptr;
        sp.wait_ns = m->step_wait_ns;
        sp.extra = m->step_extra;
        sp.trace = m->trace;
        sp.trace_n = m->trace_n;
        {
            int pc0[16] = {0};
            ProfScope prof_scope_(m, QW_PROF_STEP, pc0, st);
            if (launches) ++*launches;
            CUDA_TRY(launch_decode_step(st, sp, m->st_maps, m->num_sms));
        }
    }
    // A decode batch of >= 16 sequences runs as two halves on two streams, so that one
    // half's latency-bound projections overlap the other half's HBM-bound attention.
    // With the debug dumps on, each half writes its own rows of them (the same kernels run).
    const bool two = !engine && !prefill && !small && m->prof_kind == QW_PROF_OFF && m->split_decode && T >= 16;
    if (engine) {
        // the layers ran above
    } else if (two) {
        const int h0 = T / 2;
        CUDA_TRY(cudaEventRecord(m->ev_fork, st));
        CUDA_TRY(cudaStreamWaitEvent(m->aux_stream, m->ev_fork, 0));
        QW_TRY(run_layers(m, kv, sd, prefill, max_keys, 0, h0, st, dbg, launches, pc));
        QW_TRY(run_layers(m, kv, sd, prefill, max_keys, h0, T - h0, m->aux_stream, dbg, launches, pc));
        CUDA_TRY(cudaEventRecord(m->ev_join, m->aux_stream));
        CUDA_TRY(cudaStreamWaitEvent(st, m->ev_join, 0));
    } else {
        QW_TRY(run_layers(m, kv, sd, prefill, max_keys, 0, T, st, dbg, launches, pc));
    }
    LaunchCtx lc = {st, false, launches};  // the head follows a full dependency on the layers
    const bool pdl_on = m->pdl && m->prof_kind == QW_PROF_OFF;
#define PROF(kind) ProfScope prof_scope_(m, kind, pc, st)
    // --- final norm + tied LM head + greedy argmax (Paso 8) ---
    // The GEMV reads the 311 MB head at full bandwidth for 1-3 rows; from 4 rows on its dot
    // products cost more than the tensor-core GEMM, which streams the head once for any B.
    if (B < kLmGemmMinRows) {
        PROF(QW_PROF_LMHEAD);
        const bool d1 = !engine && dec1_step(m, sd, prefill, max_keys);  // x + the last down_proj partials
        if (d1) lc.pdl = pdl_on;
        if (B == 1 && lmhead1_ok(D, c.vocab)) {
            // the head's last CTA also ends the step (id, length): no finalize launch
            CUDA_TRY(launch_lmhead1(lc, m->x, m->last, m->fnorm, c.rms_eps, m->embed, c.vocab, D, logits, m->best,
                                    d1 ? m->d1_dpart + (size_t)((c.n_layers - 1) & 1) * dec1_parts() * D : nullptr,
                                    d1 ? dec1_parts() : 0, m->status, m->num_sms, next, kvv.len, sd.seq[0],
                                    sd.start[1] - sd.start[0], m->lm_done));
            return QW_OK;
        }
        CUDA_TRY(launch_gemv_lmhead(lc, B, m->x, m->last, m->fnorm, c.rms_eps, m->embed, c.vocab, D, logits,
                                    m->best,
                                    d1 ? m->d1_dpart + (size_t)((c.n_layers - 1) & 1) * dec1_parts() * D : nullptr,
                                    d1 ? dec1_parts() : 0));
    } else {
        {
            PROF(QW_PROF_RMSNORM);
            CUDA_TRY(launch_rmsnorm(lc, m->x, m->last, B, D, m->fnorm, c.rms_eps, m->h));
        }
        lc.pdl = pdl_on;
        PROF(QW_PROF_LMHEAD);
        GemmArgs g = {};
        g.tmA = &m->tm_embed; g.tmB = m->tm_h;
        g.a_row0 = 0; g.M = c.vocab; g.K = D; g.T = B;
        g.logits = logits; g.ld_out = c.vocab; g.best = m->best; g.status = m->status; g.num_sms = m->num_sms;
        CUDA_TRY(launch_gemm_tc(lc, EPI_ARGMAX, g));
    }
    lc.pdl = pdl_on;
    CUDA_TRY(launch_finalize(lc, sd, m->best, next, kvv));
#undef PROF
    return QW_OK;
}

static qw_status check_batch(const qw_model* m, const qw_kv* kv, int B, const int* seq_ids) {
    if (!m || !kv) return fail(QW_ERR_INVALID_ARG, "model or kv is NULL");
    if (kv->m != m) return fail(QW_ERR_INVALID_ARG, "kv belongs to another model");
    if (B < 1 || B > m->cfg.max_batch) return fail(QW_ERR_INVALID_ARG, "B=%d outside [1, max_batch]", B);
    if (!seq_ids) return fail(QW_ERR_INVALID_ARG, "seq_ids is NULL");
    std::set<int> seen;
    for (int b = 0; b < B; ++b) {
        const int s = seq_ids[b];
        if (s < 0 || s >= kv->max_seqs) return fail(QW_ERR_INVALID_ARG, "seq id %d out of range", s);
        if (!seen.insert(s).second) return fail(QW_ERR_INVALID_ARG, "seq id %d repeated", s);
    }
    return QW_OK;
}

extern "C" qw_status qw_prefill(qw_model* m, qw_kv* kv, int B, const int* seq_ids, const int* lens,
                                const int32_t* dev_token_ids, float* dev_logits, int32_t* dev_next_ids,
                                void* stream_) {
    QW_TRY(check_batch(m, kv, B, seq_ids));
    if (!lens || !dev_token_ids || !dev_next_ids) return fail(QW_ERR_INVALID_ARG, "NULL argument");
    StepDesc sd = {};
    sd.B = B;
    long long total = 0;
    int max_keys = 0;
    for (int b = 0; b < B; ++b) {
        const int s = seq_ids[b];
        if (lens[b] < 1) return fail(QW_ERR_INVALID_ARG, "lens[%d] = %d < 1", b, lens[b]);
        // the prompt continues the sequence's cache (chunked prefill): positions kv->len[s] ..
        const long long keys = (long long)kv->len[s] + lens[b];
        if (keys > m->cfg.max_context) return fail(QW_ERR_INVALID_ARG, "cache + prompt longer than max_context");
        if ((long long)kv->pt[s].size() * 16 < keys)
            return fail(QW_ERR_KV_FULL, "sequence %d reserved for %zu tokens < %lld", s, kv->pt[s].size() * 16, keys);
        sd.seq[b] = s;
        sd.start[b] = (int)total;
        total += lens[b];
        max_keys = std::max(max_keys, (int)keys);
    }
    if (total > m->cfg.max_tokens) return fail(QW_ERR_INVALID_ARG, "%lld tokens > max_tokens", total);
    sd.start[B] = (int)total;
    sd.T = (int)total;
    int launches = 0;
    QW_TRY(run_step(m, kv, sd, true, max_keys, dev_token_ids, dev_logits, dev_next_ids, (cudaStream_t)stream_,
                    true, &launches));
    m->last_launches = launches;
    for (int b = 0; b < B; ++b) kv->len[seq_ids[b]] += lens[b];
    return QW_OK;
}

// Checks a decode batch whose sequences each take n_steps more tokens; fills sd (one token
// per sequence) and the largest reserved capacity of the batch.
static qw_status decode_prepare(qw_model* m, qw_kv* kv, int B, const int* seq_ids, int n_steps, StepDesc& sd,
                                int& cap) {
    QW_TRY(check_batch(m, kv, B, seq_ids));
    if (B > m->cfg.max_tokens) return fail(QW_ERR_INVALID_ARG, "B > max_tokens");
    sd = StepDesc{};
    sd.B = B;
    sd.T = B;
    cap = 0;
    for (int b = 0; b < B; ++b) {
        const int s = seq_ids[b];
        const int capacity = std::min((int)kv->pt[s].size() * 16, m->cfg.max_context);
        if ((long long)kv->len[s] + n_steps > capacity)
            return fail(QW_ERR_KV_FULL, "sequence %d has no reserved slot for position %d", s,
                        std::max(kv->len[s], capacity));
        sd.seq[b] = s;
        sd.start[b] = b;
        cap = std::max(cap, capacity);
    }
    sd.start[B] = B;
    return QW_OK;
}

// n_steps decode steps replayed from one CUDA graph: step i reads its tokens from
// tokens_i = (i == 0 ? tokens : next + (i - 1) * next_stride) and writes its picks to
// next + i * next_stride (next_stride 0: every step in place); the last step writes logits.
// Each step begins with a kernel launched without programmatic overlap, so a step's kernels
// may read what earlier steps wrote before their dependency wait, as in separate graphs.
static qw_status decode_graph(qw_model* m, qw_kv* kv, const StepDesc& sd, int cap, int n_steps,
                              const int32_t* tokens, float* logits, int32_t* next, int next_stride,
                              cudaStream_t st) {
    const int B = sd.B;
    // graph key: everything baked into the captured kernels
    const SplitPlan sp = plan_splits(m, B, cap);
    std::vector<long long> key;
    key.reserve(B + 20);
    key.push_back(B);
    key.push_back(cap);
    key.push_back(n_steps);
    key.push_back(next_stride);
    key.push_back((long long)(uintptr_t)tokens);
    key.push_back((long long)(uintptr_t)logits);
    key.push_back((long long)(uintptr_t)next);
    key.push_back((long long)(uintptr_t)kv);
    key.push_back(sp.chunk);
    key.push_back(m->prof_kind);
    key.push_back(m->pdl ? 1 : 0);
    key.push_back(m->split_decode ? 1 : 0);
    key.push_back(m->use_step ? m->step_gp : 0);
    key.push_back((long long)m->step_wait_ns);
    key.push_back(m->step_extra);
    key.push_back(m->use_dec1 ? 1 : 0);
    key.push_back(m->prof_kind || m->trace ? (long long)m->prof_gen : 0);
    for (int b = 0; b < B; ++b) key.push_back(sd.seq[b]);
    auto it = m->graphs.find(key);
    if (it == m->graphs.end()) {
        if (m->graphs.size() >= 64) {  // evict the least recently used entry
            auto lru = m->graphs.begin();
            for (auto jt = m->graphs.begin(); jt != m->graphs.end(); ++jt)
                if (jt->second.last_use < lru->second.last_use) lru = jt;
            cudaGraphExecDestroy(lru->second.exec);
            m->graphs.erase(lru);
        }
        int launches = 0;
        cudaGraph_t graph = nullptr;
        CUDA_TRY(cudaStreamBeginCapture(m->cap_stream, cudaStreamCaptureModeThreadLocal));
        qw_status s = QW_OK;
        for (int i = 0; i < n_steps && s == QW_OK; ++i) {
            m->chain_step = i > 0;
            s = run_step(m, kv, sd, false, cap, i == 0 ? tokens : next + (size_t)(i - 1) * next_stride,
                         i == n_steps - 1 ? logits : nullptr, next + (size_t)i * next_stride, m->cap_stream, false,
                         &launches);
        }
        m->chain_step = false;
        cudaError_t e = cudaStreamEndCapture(m->cap_stream, &graph);
        if (s != QW_OK) {
            if (graph) cudaGraphDestroy(graph);
            return s;
        }
        if (e != cudaSuccess) return fail(QW_ERR_CUDA, "graph capture failed: %s", cudaGetErrorString(e));
        cudaGraphExec_t exec = nullptr;
        e = cudaGraphInstantiate(&exec, graph, 0);
        cudaGraphDestroy(graph);
        if (e != cudaSuccess) return fail(QW_ERR_CUDA, "graph instantiate failed: %s", cudaGetErrorString(e));
        it = m->graphs.emplace(key, GraphEntry{exec, launches, 0}).first;
    }
    it->second.last_use = ++m->use_clock;
    CUDA_TRY(cudaGraphLaunch(it->second.exec, st));
    m->last_launches = it->second.launches;
    for (int b = 0; b < B; ++b) kv->len[sd.seq[b]] += n_steps;
    return QW_OK;
}

extern "C" qw_status qw_decode_step(qw_model* m, qw_kv* kv, int B, const int* seq_ids,
                                    const int32_t* dev_token_ids, float* dev_logits, int32_t* dev_next_ids,
                                    void* stream_) {
    if (!dev_token_ids || !dev_next_ids) return fail(QW_ERR_INVALID_ARG, "NULL argument");
    StepDesc sd;
    int cap = 0;
    QW_TRY(decode_prepare(m, kv, B, seq_ids, 1, sd, cap));
    cudaStream_t st = (cudaStream_t)stream_;
    if (m->dbg_hidden) {
        int launches = 0;
        int max_keys = 0;
        for (int b = 0; b < B; ++b) max_keys = std::max(max_keys, kv->len[seq_ids[b]] + 1);
        QW_TRY(run_step(m, kv, sd, false, max_keys, dev_token_ids, dev_logits, dev_next_ids, st, true, &launches));
        m->last_launches = launches;
        for (int b = 0; b < B; ++b) kv->len[seq_ids[b]] += 1;
        return QW_OK;
    }
    return decode_graph(m, kv, sd, cap, 1, dev_token_ids, dev_logits, dev_next_ids, 0, st);
}

extern "C" qw_status qw_decode_steps(qw_model* m, qw_kv* kv, int B, const int* seq_ids, int n_steps,
                                     const int32_t* dev_token_ids, int32_t* dev_out_ids, void* stream_) {
    if (!dev_token_ids || !dev_out_ids) return fail(QW_ERR_INVALID_ARG, "NULL argument");
    if (n_steps < 1 || n_steps > QW_MAX_GRAPH_STEPS)
        return fail(QW_ERR_INVALID_ARG, "n_steps %d outside [1, %d]", n_steps, QW_MAX_GRAPH_STEPS);
    StepDesc sd;
    int cap = 0;
    QW_TRY(decode_prepare(m, kv, B, seq_ids, n_steps, sd, cap));
    cudaStream_t st = (cudaStream_t)stream_;
    if (m->dbg_hidden || m->prof_kind || m->trace) {
        // the debug dumps, profiling events and trace records describe one step: step by step
        int total = 0;
        for (int i = 0; i < n_steps; ++i) {
            QW_TRY(qw_decode_step(m, kv, B, seq_ids, i == 0 ? dev_token_ids : dev_out_ids + (size_t)(i - 1) * B,
                                  nullptr, dev_out_ids + (size_t)i * B, stream_));
            total += m->last_launches;
        }
        m->last_launches = total;
        return QW_OK;
    }
    return decode_graph(m, kv, sd, cap, n_steps, dev_token_ids, nullptr, dev_out_ids, B, st);
}

// Paso 9 over a batch: prefill, then decode steps feeding each pick back on the device. With
// eos_id >= 0 a sequence stops after its first pick equal to eos_id (the pick is kept, never
// fed). Stopped sequences keep stepping with the rest of the batch (one graph for the whole
// batch); their extra positions are dropped from the cache at the end. The host looks at the
// picks every kEosCheck steps and ends the loop once every sequence has stopped.
static qw_status generate_impl(qw_model* m, qw_kv* kv, int B, const int* seq_ids, const int* lens,
                               const int32_t* host_prompt_ids, int n_decode, int eos_id, int32_t* host_out_ids,
                               int32_t* host_out_counts, cudaStream_t st) {
    constexpr int kEosCheck = 8;
    QW_TRY(check_batch(m, kv, B, seq_ids));
    if (!lens || !host_prompt_ids || !host_out_ids) return fail(QW_ERR_INVALID_ARG, "NULL argument");
    if (n_decode < 0 || n_decode + 1 > m->cfg.max_context) return fail(QW_ERR_INVALID_ARG, "n_decode out of range");
    long long total = 0;
    for (int b = 0; b < B; ++b) {
        if (lens[b] < 1) return fail(QW_ERR_INVALID_ARG, "lens[%d] < 1", b);
        const int s = seq_ids[b];
        if (kv->len[s] != 0) return fail(QW_ERR_BAD_STATE, "generate needs empty sequences (%d is not)", s);
        // every position the loop writes must fit the context, or a decode step would fail
        // after the prefill has already advanced the cache
        if ((long long)lens[b] + n_decode > m->cfg.max_context)
            return fail(QW_ERR_INVALID_ARG, "sequence %d: prompt %d + %d decode tokens > max_context %d", s, lens[b],
                        n_decode, m->cfg.max_context);
        if ((long long)kv->pt[s].size() * 16 < (long long)lens[b] + n_decode)
            return fail(QW_ERR_KV_FULL, "sequence %d not reserved for prompt + %d decode tokens", s, n_decode);
        total += lens[b];
    }
    if (total > m->cfg.max_tokens) return fail(QW_ERR_INVALID_ARG, "prompts exceed max_tokens");
    CUDA_TRY(cudaMemcpyAsync(m->gen_tok, host_prompt_ids, (size_t)total * 4, cudaMemcpyHostToDevice, st));
    QW_TRY(qw_prefill(m, kv, B, seq_ids, lens, m->gen_tok, nullptr, m->gen_out, st));
    int launches = m->last_launches;
    std::vector<int32_t> tmp((size_t)(n_decode + 1) * B);
    std::vector<int> stop_at(B, -1);  // index of a sequence's first EOS pick
    int n_stopped = 0, seen = 0;      // picks [0, seen) were read on the host
    auto look = [&](int upto) -> qw_status {  // read picks [seen, upto] and note the stops
        if (upto < seen) return QW_OK;
        CUDA_TRY(cudaMemcpyAsync(tmp.data() + (size_t)seen * B, m->gen_out + (size_t)seen * B,
                                 (size_t)(upto + 1 - seen) * B * 4, cudaMemcpyDeviceToHost, st));
        CUDA_TRY(cudaStreamSynchronize(st));
        for (int i = seen; i <= upto; ++i)
            for (int b = 0; b < B; ++b)
                if (eos_id >= 0 && stop_at[b] < 0 && tmp[(size_t)i * B + b] == eos_id) {
                    stop_at[b] = i;
                    ++n_stopped;
                }
        seen = upto + 1;
        return QW_OK;
    };
    if (eos_id >= 0) QW_TRY(look(0));
    // picks i = 1 .. n_decode: each chunk of steps is one graph that feeds row i - 1 of gen_out
    // and writes row i (chunks of kEosCheck steps with an EOS, so the host can stop early; for
    // more than 8 sequences, whose steps are hundreds of launches each, chunks of kEosCheck too,
    // which keeps each graph to a few thousand nodes)
    int last = 0;
    const int chunk = eos_id >= 0 || B > 8 ? kEosCheck : QW_MAX_GRAPH_STEPS;
    while (last < n_decode && n_stopped < B) {
        const int n = std::min(chunk, n_decode - last);
        QW_TRY(qw_decode_steps(m, kv, B, seq_ids, n, m->gen_out + (size_t)last * B, m->gen_out + (size_t)(last + 1) * B,
                               st));
        launches += m->last_launches;
        last += n;
        if (eos_id >= 0) QW_TRY(look(last));
    }
    QW_TRY(look(last));
    for (int b = 0; b < B; ++b) {
        const int n = stop_at[b] >= 0 ? stop_at[b] + 1 : last + 1;
        for (int i = 0; i <= n_decode; ++i)
            host_out_ids[(size_t)b * (n_decode + 1) + i] = i < n ? tmp[(size_t)i * B + b] : -1;
        if (host_out_counts) host_out_counts[b] = n;
        // fed: the prompt and the picks before the stop; the cache advanced once per step
        if (stop_at[b] >= 0 && stop_at[b] < last) QW_TRY(qw_kv_truncate(kv, seq_ids[b], lens[b] + stop_at[b], st));
    }
    CUDA_TRY(cudaStreamSynchronize(st));
    m->last_launches = launches;
    return QW_OK;
}

extern "C" qw_status qw_generate(qw_model* m, qw_kv* kv, int B, const int* seq_ids, const int* lens,
                                 const int32_t* host_prompt_ids, int n_decode, int32_t* host_out_ids,
                                 void* stream_) {
    return generate_impl(m, kv, B, seq_ids, lens, host_prompt_ids, n_decode, -1, host_out_ids, nullptr,
                         (cudaStream_t)stream_);
}

extern "C" qw_status qw_generate_eos(qw_model* m, qw_kv* kv, int B, const int* seq_ids, const int* lens,
                                     const int32_t* host_prompt_ids, int n_decode, int eos_id,
                                     int32_t* host_out_ids, int32_t* host_out_counts, void* stream_) {
    if (eos_id < 0 || (m && eos_id >= m->cfg.vocab)) return fail(QW_ERR_INVALID_ARG, "eos_id outside [0, vocab)");
    if (!host_out_counts) return fail(QW_ERR_INVALID_ARG, "NULL argument");
    return generate_impl(m, kv, B, seq_ids, lens, host_prompt_ids, n_decode, eos_id, host_out_ids, host_out_counts,
                         (cudaStream_t)stream_);
}

extern "C" qw_status qw_sync_status(qw_model* m, void* stream_) {
    if (!m) return fail(QW_ERR_INVALID_ARG, "model is NULL");
    cudaStream_t st = (cudaStream_t)stream_;
    CUDA_TRY(cudaStreamSynchronize(st));
    int word = 0;
    CUDA_TRY(cudaMemcpy(&word, m->status, 4, cudaMemcpyDeviceToHost));
    CUDA_TRY(cudaMemset(m->status, 0, 4));
    CUDA_TRY(cudaMemset(m->st_abort, 0, 4));
    if (word & QW_DEV_TIMEOUT) {
        // a kernel that gave up may have left arrival tickets behind
        CUDA_TRY(cudaMemset(m->st_tick, 0, (size_t)2 * step_tiles(m->cfg.hidden, m->cfg.inter, m->qkv_rows) * 4));
        CUDA_TRY(cudaMemset(m->counters, 0, (size_t)m->L.part_T * m->cfg.n_kv_heads * 4));
    }
    if (word & QW_DEV_BAD_TOKEN) return fail(QW_ERR_BAD_TOKEN, "a token id was outside [0, vocab)");
    if (word & QW_DEV_BAD_POS) return fail(QW_ERR_BAD_POS, "a position had no reserved page");
    if (word & QW_DEV_TIMEOUT) return fail(QW_ERR_TIMEOUT, "a bounded wait in a kernel timed out");
    if (word & QW_DEV_RANGE)
        return fail(QW_ERR_RANGE, "an activation or K/V value stored as fp16 was outside its range (|v| > 65504)");
    return QW_OK;
}
