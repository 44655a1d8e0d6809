/*
 * qw.h - C ABI of the GB300 (sm_103a) Qwen3-style decoder library (libqw.so).
 *
 * The library runs the decoder forward pass walked through on the page "Dentro de un LLM:
 * Inferencia en Python puro para Qwen3-0.6B en MLX": embedding gather (Paso 2), RMSNorm
 * (Paso 3), Q/K/V projections with per-head QK-norm and rotate-half RoPE (Pasos 4-5), KV
 * cache append and grouped-query causal attention (Paso 5), o_proj, SwiGLU (Paso 6), the
 * residual block (Paso 7), final norm + tied LM head + greedy argmax (Paso 8), and the
 * prefill / decode loop (Paso 9).
 *
 * Conventions shared by every entry point:
 *  - Device pointers are CUDA device addresses owned by the CALLER. The library never
 *    allocates device memory; it carves what it needs from the workspace and KV pool the
 *    caller hands it. Borrowed buffers must outlive the object that borrows them.
 *  - Host pointers are plain host memory, read during the call only (never retained).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream). Work is
 *    enqueued asynchronously on it unless the function says it synchronises.
 *  - Every call returns QW_OK (0) or a negative qw_status. An error found on the host is
 *    reported before anything is enqueued and leaves all state unchanged. qw_last_error()
 *    returns a message for the calling thread's last error.
 *  - Errors found on the device (a token id out of range, a position without a reserved
 *    page, a wait that timed out) set bits in a device status word; the affected rows are
 *    written as zeros and nothing traps. qw_sync_status() reads and clears that word.
 *  - Weights are given as bf16 in the HF [out_features, in_features] row-major layout
 *    (x @ W^T). The projection matrices are packed as fp16 copies, the operand type of the
 *    tensor cores here: fp16 holds every bf16 value of magnitude in [2^-14, 65504] exactly
 *    and rounds smaller ones to its subnormal grid (error <= 2^-25). Activations that feed
 *    a matrix product and the KV cache are fp16; the residual stream, accumulators,
 *    norms, softmax and logits are fp32.
 */
#ifndef QW_H
#define QW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QW_OK = 0,
    QW_ERR_INVALID_ARG = -1, /* a null/misaligned pointer, a size or id out of range          */
    QW_ERR_KV_FULL = -2,     /* not enough free pages, or a sequence past its reservation      */
    QW_ERR_BAD_STATE = -3,   /* e.g. generate into a non-empty sequence, quantize twice       */
    QW_ERR_CUDA = -4,        /* a CUDA runtime call failed (message has the CUDA error)        */
    QW_ERR_BAD_TOKEN = -5,   /* device status: a token id outside [0, vocab)                  */
    QW_ERR_TIMEOUT = -6,     /* device status: a bounded wait inside a kernel gave up          */
    QW_ERR_UNSUPPORTED = -7, /* a shape this build has no kernel for                          */
    QW_ERR_BAD_POS = -8,     /* device status: a position with no page in the page table      */
    QW_ERR_RANGE = -9        /* device status: an activation or K/V value stored as fp16 was
                              * beyond the fp16 range (|v| > 65504, or NaN)                    */
} qw_status;

/* Model shape. Per-layer dims of Qwen3-0.6B: hidden 1024, 16 query / 8 KV heads of 128,
 * SwiGLU 3072, vocab 151936, 28 layers, eps 1e-6, theta 1e6 (Pasos 2-7). This build
 * supports head_dim 128, n_heads == 2 * n_kv_heads, hidden % 256 == 0, inter % 256 == 0,
 * (n_heads * head_dim) % 256 == 0, vocab % 128 == 0, page_size 16, tie_embed 1. */
typedef struct {
    int n_layers;
    int hidden;
    int n_heads;
    int n_kv_heads;
    int head_dim;
    int inter;
    int vocab;
    int page_size;   /* tokens per KV page; 16                                            */
    int tie_embed;   /* 1: the LM head is model.embed_tokens.weight (Paso 8, tied)        */
    float rms_eps;   /* 1e-6 (Paso 3)                                                     */
    double rope_theta; /* 1e6 (Paso 4)                                                    */
    int max_tokens;  /* most tokens one prefill/decode call may carry (sizes workspace)   */
    int max_batch;   /* most sequences in one call (<= QW_MAX_BATCH)                      */
    int max_context; /* longest sequence in tokens (RoPE table and page-table rows)       */
} qw_config;

#define QW_MAX_BATCH 256

/* Device pointers of one decoder layer's bf16 tensors, HF names. */
typedef struct {
    const void* input_layernorm;          /* [hidden]                        */
    const void* q_proj;                   /* [n_heads*head_dim, hidden]      */
    const void* k_proj;                   /* [n_kv_heads*head_dim, hidden]   */
    const void* v_proj;                   /* [n_kv_heads*head_dim, hidden]   */
    const void* o_proj;                   /* [hidden, n_heads*head_dim]      */
    const void* q_norm;                   /* [head_dim], shared by all heads */
    const void* k_norm;                   /* [head_dim]                      */
    const void* post_attention_layernorm; /* [hidden]                        */
    const void* gate_proj;                /* [inter, hidden]                 */
    const void* up_proj;                  /* [inter, hidden]                 */
    const void* down_proj;                /* [hidden, inter]                 */
} qw_layer_ptrs;

typedef struct {
    const void* embed_tokens;     /* [vocab, hidden]; BORROWED for the model's lifetime   */
    const void* norm;             /* [hidden] final norm                                  */
    const qw_layer_ptrs* layers;  /* host array of n_layers entries                       */
} qw_weight_ptrs;

typedef struct qw_model qw_model;
typedef struct qw_kv qw_kv;

/* Bytes of device workspace qw_init_weights needs for `cfg` (fp16 packed weights and an
 * fp16 copy of the embedding for the LM head, RoPE table, activations for max_tokens,
 * split-KV partials, status word). 0 if cfg is invalid. */
size_t qw_model_workspace_bytes(const qw_config* cfg);

/* Validate cfg, pack the weights into `dev_workspace` (fp16 copies of the matrices with
 * q|k|v rows concatenated per layer, norm weights copied as bf16), build the fp32 RoPE
 * cos/sin table (host fp64, Paso 4) and carve the activation buffers. Synchronises
 * `stream`; the source tensors may be freed afterwards except embed_tokens, which the
 * embedding gather keeps reading and must outlive the model. A weight beyond the fp16 range,
 * or a norm weight above 65504 / sqrt(n) (n = hidden for the layer and final norms, head_dim
 * for the QK-norms; it would let a normalised fp16 operand overflow), gives
 * QW_ERR_INVALID_ARG. ws_bytes >= qw_model_workspace_bytes(cfg), workspace 256-byte
 * aligned. On success *out owns host state only. */
qw_status qw_init_weights(const qw_config* cfg, const qw_weight_ptrs* w, void* dev_workspace,
                          size_t ws_bytes, void* stream, qw_model** out);

/* Bytes of device pool for a paged KV cache of `n_pages` pages of page_size tokens for
 * `max_seqs` sequences: per-sequence lengths and page tables, then K and V pools laid out
 * [n_layers][n_pages][n_kv_heads][page_size][head_dim] fp16. */
size_t qw_kv_pool_bytes(const qw_model* m, int n_pages, int max_seqs);

/* Bind a caller-owned pool (256-byte aligned) as the KV cache (Paso 5, "KV cache"). The page
 * count is the largest that fits pool_bytes. Zeroes lengths and page tables on `stream`. */
qw_status qw_kv_alloc(qw_model* m, void* dev_pool, size_t pool_bytes, int max_seqs, void* stream,
                      qw_kv** out);

/* Make sure sequence `seq_id` owns pages for `total_tokens` positions, taking free pages
 * lowest id first (QW_ERR_KV_FULL, nothing taken, if too few are free). Page-table rows are
 * written on `stream`. */
qw_status qw_kv_reserve(qw_kv* kv, int seq_id, int total_tokens, void* stream);

/* Free the pages of `seq_id` (-1: every sequence) and set its length to 0, on `stream`. */
qw_status qw_kv_reset(qw_kv* kv, int seq_id, void* stream);

/* Keep only the first n_tokens positions of sequence seq_id (n_tokens <= its length): the
 * length goes back to n_tokens, the pages stay reserved, and later steps overwrite the
 * dropped positions. Written on `stream`. */
qw_status qw_kv_truncate(qw_kv* kv, int seq_id, int n_tokens, void* stream);

int qw_kv_free_pages(const qw_kv* kv);
int qw_kv_length(const qw_kv* kv, int seq_id); /* host mirror of the device length */

/* Prefill (Paso 9, first forward): run B sequences' prompts through the model. A prompt
 * continues its sequence's cache (chunked prefill): its tokens take positions len .. len +
 * lens[b] - 1 after the sequence's current length len (0 for a first prompt) and attend to the
 * cached prefix and to the earlier prompt tokens (causal by position).
 * seq_ids[B], lens[B] (host): sequence ids and prompt lengths (each >= 1; each sequence
 * reserved for at least len + lens[b] tokens, at most max_context). dev_token_ids: the
 * prompts concatenated, sum(lens) int32. dev_logits: [B, vocab] fp32 logits of each prompt's
 * last position, or NULL. dev_next_ids: [B] int32 greedy picks (argmax, lowest index on
 * ties). Appends every prompt token's K/V to the cache and advances the lengths. */
qw_status qw_prefill(qw_model* m, qw_kv* kv, int B, const int* seq_ids, const int* lens,
                     const int32_t* dev_token_ids, float* dev_logits, int32_t* dev_next_ids,
                     void* stream);

/* One decode step (Paso 9 loop body): each of the B sequences takes one new token at
 * position = its current length. dev_token_ids [B] may alias the previous step's
 * dev_next_ids. Outputs as in qw_prefill. The step is replayed from a CUDA graph cached per
 * (B, seq_ids, pointers); the first call with a new key captures it. */
qw_status qw_decode_step(qw_model* m, qw_kv* kv, int B, const int* seq_ids,
                         const int32_t* dev_token_ids, float* dev_logits, int32_t* dev_next_ids,
                         void* stream);

/* n_steps greedy decode steps of the same B sequences (the loop of Paso 9, every pick fed
 * back on the device) replayed from ONE CUDA graph, cached per (B, seq_ids, n_steps,
 * pointers): no host work and no graph boundary between the steps. dev_token_ids [B]: the
 * tokens of the first step; dev_out_ids [n_steps, B] int32: row i holds step i's picks and
 * is step i + 1's input (dev_token_ids may be dev_out_ids - B, i.e. the row before). No
 * logits are written. Each sequence must be reserved for n_steps more tokens (else
 * QW_ERR_KV_FULL, nothing launched); 1 <= n_steps <= QW_MAX_GRAPH_STEPS (else
 * QW_ERR_INVALID_ARG). The picks, cache contents and lengths are those of n_steps calls of
 * qw_decode_step (each step starts with a full dependency on the one before). With the debug
 * dumps, profiling events or trace records set the steps run one graph each. */
#define QW_MAX_GRAPH_STEPS 64
qw_status qw_decode_steps(qw_model* m, qw_kv* kv, int B, const int* seq_ids, int n_steps,
                          const int32_t* dev_token_ids, int32_t* dev_out_ids, void* stream);

/* Greedy generation from HOST buffers (Paso 9 at temperature 0, no EOS stop): copies the
 * concatenated prompts (host_prompt_ids, sum(lens) int32) to the device, prefills, runs
 * n_decode decode steps feeding each pick back on the device, copies the picks to
 * host_out_ids ([B, n_decode + 1] int32, row b = sequence b) and synchronises `stream`.
 * Sequences must be empty and reserved for lens[b] + n_decode tokens. The decode steps run
 * as qw_decode_steps graphs of up to QW_MAX_GRAPH_STEPS steps. */
qw_status qw_generate(qw_model* m, qw_kv* kv, int B, const int* seq_ids, const int* lens,
                      const int32_t* host_prompt_ids, int n_decode, int32_t* host_out_ids,
                      void* stream);

/* Greedy generation with an EOS stop (Paso 9: the page's loop ends when a pick equals
 * EOS_ID; the page leaves the id undefined, so the caller gives it). As qw_generate, except:
 * a sequence stops after its first pick equal to eos_id, which is kept as its last output and
 * never fed to the model. Row b of host_out_ids ([B, n_decode + 1]) holds host_out_counts[b]
 * picks (up to and including that EOS; n_decode + 1 without one) followed by -1, and the
 * sequence's cache ends with the prompt and the picks it fed. The batch steps until every
 * sequence has stopped (the host reads the picks every 8 steps) or n_decode steps ran;
 * stopped sequences keep stepping with the batch meanwhile and their extra positions are
 * dropped from the cache at the end. Errors as qw_generate, plus QW_ERR_INVALID_ARG for
 * eos_id outside [0, vocab) or a NULL host_out_counts. */
qw_status qw_generate_eos(qw_model* m, qw_kv* kv, int B, const int* seq_ids, const int* lens,
                          const int32_t* host_prompt_ids, int n_decode, int eos_id, int32_t* host_out_ids,
                          int32_t* host_out_counts, void* stream);

/* Synchronise `stream`, read and clear the device status word. Returns QW_OK or the first
 * of QW_ERR_BAD_TOKEN, QW_ERR_BAD_POS, QW_ERR_TIMEOUT, QW_ERR_RANGE that the word records.
 * QW_ERR_RANGE: a value the step stores as fp16 (the attention values appended to the KV
 * cache, the SwiGLU activation, the raw q|k|v projections staged for the QK-norm) was
 * beyond the fp16 range; the outputs of that step are not valid. (The normalised operands
 * cannot overflow: qw_init_weights refuses norm weights above 65504 / sqrt(n).) */
qw_status qw_sync_status(qw_model* m, void* stream);

/* Message for the calling thread's last error ("" if none). Valid until the next call. */
const char* qw_last_error(void);

void qw_free_model(qw_model* m); /* frees host state and cached graphs; not the workspace */
void qw_free_kv(qw_kv* kv);

/* ---- Test and inspection hooks (not on the hot path) -------------------------------- */

/* When dev_hidden is non-NULL, every following prefill/decode call copies the residual
 * stream after each layer to dev_hidden[layer][t][hidden] (fp32, t < that call's token
 * count) and writes each token's position and KV slot (page * page_size + offset) to
 * dev_positions[t] / dev_slots[t]. Pass NULLs to turn it off. Calls made while it is on are
 * not graph-captured. */
qw_status qw_debug_set(qw_model* m, float* dev_hidden, int32_t* dev_positions, int32_t* dev_slots);

/* While qw_debug_set is on and dev_attn is non-NULL, prefill and decode calls also copy each
 * layer's attention output, the input of o_proj, to dev_attn[layer][t][n_heads * head_dim] (fp16,
 * t < that call's token count). NULL turns it off. */
qw_status qw_debug_set_attn(qw_model* m, void* dev_attn);

/* Copy sequence seq_id's page table (host mirror) into host_out[0..max_pages); returns the
 * number of pages it owns, or a negative qw_status. */
int qw_kv_page_table(const qw_kv* kv, int seq_id, int32_t* host_out, int max_pages);

/* Device addresses of the K and V pools ([n_layers][n_pages][n_kv_heads][page][head_dim]
 * fp16) and the page count. */
qw_status qw_kv_pool_ptrs(const qw_kv* kv, void** dev_k, void** dev_v, int* n_pages);

/* Fill positions [0, n_tokens) of sequence seq_id (reserved, empty) with synthetic K/V from
 * the counter-based SplitMix64 generator: element index
 *   idx = (((layer*2 + which) << 22 | pos) * n_kv_heads + head) * head_dim + dim,
 *   z = splitmix64(seed + (idx + 1) * 0x9E3779B97F4A7C15), b = (int8)(z >> 56),
 *   K = b / 64, V = b / 128 (exact in fp16),
 * and set the sequence's length to n_tokens. Stands in for a long prefill. */
qw_status qw_kv_fill_synthetic(qw_kv* kv, int seq_id, int n_tokens, uint64_t seed, void* stream);

/* Number of kernels the last prefill / decode call enqueued (graph replays count the
 * kernels inside the graph; a qw_decode_steps call counts all its steps). */
int qw_last_launch_count(const qw_model* m);

/* Kernel kinds for qw_profile_set. */
enum {
    QW_PROF_OFF = 0,
    QW_PROF_QKV = 1,      /* q|k|v projection (RMSNorm fused on the small-batch path)    */
    QW_PROF_ROPE = 2,     /* QK-norm + RoPE + KV append                                   */
    QW_PROF_ATTN = 3,     /* attention                                                    */
    QW_PROF_OPROJ = 4,    /* o_proj + residual                                            */
    QW_PROF_GATEUP = 5,   /* gate/up + SiLU*mul (RMSNorm fused on the small-batch path)   */
    QW_PROF_DOWN = 6,     /* down_proj + residual                                         */
    QW_PROF_LMHEAD = 7,   /* final norm + tied LM head + argmax                           */
    QW_PROF_RMSNORM = 8,  /* stand-alone RMSNorm (tensor-core path)                       */
    QW_PROF_STEP = 9      /* the decode-step kernel (every layer of a decode step)         */
};

/* Options for qw_set_option. */
enum {
    /* (option 1 is not used) */
    /* 1 (default): consecutive launches use programmatic dependent launch. */
    QW_OPT_PDL = 2,
    /* 1 (default): a decode step of >= 16 sequences runs as two halves on two streams whose
     * kernels overlap (each half's projections run while the other half's attention reads
     * the KV cache); 0: one chain. Results agree within rounding (the attention's key split
     * depends on the batch size). Not used for steps the decode-step kernel runs. */
    QW_OPT_SPLIT_DECODE = 3,
    /* 1 (where the shape allows it and one 256-thread CTA per SM fits; default 0): the layers of
     * a decode step of 16 .. 64 sequences run as ONE cooperative kernel -- the batch as two
     * halves, projection CTAs (tcgen05 GEMMs with weights streamed ahead) and attention CTAs
     * ordered by counters in global memory, so one half's projections overlap the other
     * half's attention without kernel boundaries; 0: the launch-per-phase path. Both compute
     * the same operations; results agree within rounding. */
    QW_OPT_DECODE_STEP_KERNEL = 4,
    /* CTAs given to the projection role of the decode-step kernel (default min(64, SMs / 2));
     * the rest run attention. Valid: 1 .. SMs - 1. */
    QW_OPT_STEP_PROJ_CTAS = 5,
    /* Bound, in microseconds, of every wait of the decode-step kernel on another CTA (default
     * 2,000,000). When a wait runs out the kernel sets QW_ERR_TIMEOUT in the status word, every
     * CTA stops, and qw_sync_status reports it and clears the kernel's counters. For tests. */
    QW_OPT_TEST_WAIT_LIMIT_US = 6,
    /* Test only: the first o_proj unit of the decode-step kernel waits for this many arrivals
     * more than the attention provides (default 0), so that its wait runs out. */
    QW_OPT_TEST_EXTRA_ARRIVALS = 7,
    /* 1 (default where available: hidden 1024, inter 2048/3072/4096, n_kv_heads <= 8, more
     * than one layer, and the device fits the kernels' 16- and 8-CTA clusters): a decode step of ONE token with
     * bf16 weights over a
     * cache of at most 128 keys runs each layer as two cluster launches -- (RMSNorm, q|k|v,
     * QK-norm, RoPE, KV append, attention, o_proj) and (RMSNorm, gate/up, SwiGLU, down_proj),
     * with the exchanges inside a layer through distributed shared memory; 0: the
     * launch-per-phase path. Both compute the same operations; results agree within rounding. */
    QW_OPT_BATCH1_CLUSTERS = 8
};
qw_status qw_set_option(qw_model* m, int option, int value);

/* Inspection (%globaltimer values, ns, uint64) while dev_buf is non-NULL; NULL turns it off.
 * Decode-step kernel (QW_OPT_DECODE_STEP_KERNEL): CTA c writes up to per_cta records of 8
 * values at dev_buf[(c * per_cta + k) * 8] (record id, then its phase times).
 * Batch-1 decode steps on the cluster path (QW_OPT_BATCH1_CLUSTERS) write, for layer l, launch
 * k (0: attention kernel, 1: MLP kernel) and CTA c < 128, eight values at
 * dev_buf[((2l + k) * 128 + c) * 8]: entry, weights issued, dependency wait over, x staged,
 * then three points of the kernel's phases, and exit (per_cta is not used; the buffer holds
 * n_layers * 2048 values). NULL turns it off. */
qw_status qw_trace_set(qw_model* m, unsigned long long* dev_buf, int per_cta);

/* Bracket the j-th launch of kernel kind `kind` in every following prefill/decode call with
 * cudaEventRecord(events[2j]) before and cudaEventRecord(events[2j+1]) after it, on the
 * launching stream (captured as event-record nodes in decode graphs), for 2j+1 < n_events.
 * `events` are caller-owned cudaEvent_t handles (timing enabled) that must outlive every
 * graph captured while they are set; kind QW_PROF_OFF (or events NULL) turns it off. */
qw_status qw_profile_set(qw_model* m, int kind, void* const* events, int n_events);

/* ---- Weight-only quantization ("Lo que omite el script": 4- and 8-bit weights) --------- */

/* Bytes of the caller-owned device buffer that qw_quantize_weights needs for `bits` (8 or 4);
 * 0 for other values. */
size_t qw_quantize_bytes(const qw_model* m, int bits);

/* Quantizes the projections of every layer (q|k|v, o_proj, gate, up, down; not the norms and
 * not the tied embedding / LM head) to grouped affine codes: groups of 64 inputs, scale =
 * (max - min) / (2^bits - 1) and bias = min per group computed in fp32 and stored as fp16,
 * code = clamp(rint((w - bias) / scale), 0, 2^bits - 1) (0 where the fp16 scale is 0),
 * weight = scale * code + bias. The codes and (scale, bias) words go to dev_buf (256-byte
 * aligned, at least qw_quantize_bytes(m, bits), owned by the caller, kept alive as long as the
 * model is used). From then on the small-batch paths (<= 8 token rows) read the codes, and
 * the tensor-core paths use the dequantized weights (written over the model's fp16 copies),
 * so every call computes with the same quantized model. Irreversible for this model handle.
 * Asynchronous on `stream`. Errors: QW_ERR_INVALID_ARG (bits, buffer), QW_ERR_BAD_STATE
 * (already quantized), QW_ERR_UNSUPPORTED (a shape
 * other than hidden 1024 with o_proj / down_proj inputs of 2048 or 3072). */
qw_status qw_quantize_weights(qw_model* m, int bits, void* dev_buf, size_t bytes, void* stream);

/* ---- Sampling (Paso 8) ------------------------------------------------------------------ */

/* Temperature + top-p sampling of B rows of logits, one token per row: row b is
 * dev_logits[b * ld + v], v < vocab (fp32; e.g. the logits a prefill or decode call wrote),
 * and its token goes to dev_next_ids[b].
 * temperature == 0: greedy argmax, lowest index on ties (dev_uniform may be NULL).
 * temperature > 0: p = softmax(logits / temperature); the nucleus is the shortest prefix of
 * the probabilities in descending order (equal values by ascending token id) whose running
 * sum reaches top_p, i.e. one more token than the running sums below top_p; the token is
 * drawn by inverse CDF from dev_uniform[b] in [0, 1) (values outside are clamped): the kept
 * tokens are enumerated by ascending token id and the first whose running kept probability
 * exceeds u times the kept total is chosen. The running sums are exact sums of the fp32
 * probabilities rounded to multiples of 2^-40, so the result is deterministic.
 * Asynchronous on `stream`; every buffer belongs to the caller; one cluster of 8 CTAs per
 * row, each CTA holding an eighth of the row in shared memory. Errors (nothing enqueued):
 * QW_ERR_INVALID_ARG for B outside [1, 65535], vocab outside [1, 196608], ld < vocab, a NULL
 * buffer, a negative or non-finite temperature, top_p outside (0, 1]. */
qw_status qw_sample_top_p(int B, int vocab, const float* dev_logits, size_t ld, float temperature, float top_p,
                          const float* dev_uniform, int32_t* dev_next_ids, void* stream);

/* ---- For callers that cannot allocate device memory ---------------------------------- */

/* The page has no counterpart to this entry point; it serves callers that must not call
 * cudaMalloc at the point of use: code running under another framework's fixed device
 * budget, serving loops that never touch the allocator after start-up, or code that
 * prepares work while a stream is being captured.
 *
 * Final RMSNorm + tied LM head + greedy argmax (the same kernel as the small-batch path of
 * qw_prefill / qw_decode_step) over B caller-provided fp32 residual rows dev_x [B, hidden]
 * (16-byte aligned): writes dev_logits [B, vocab] fp32 (or skips it when NULL) and
 * dev_next_ids [B] (lowest index on ties), asynchronously on `stream`. It allocates
 * nothing (no cudaMalloc, cudaFree or allocating library call): its only scratch, B
 * packed 64-bit argmax keys, is a file-scope device array of QW_NOALLOC_MAX_ROWS entries
 * that every GPU loading the library holds until exit. B > QW_NOALLOC_MAX_ROWS gives
 * QW_ERR_INVALID_ARG. The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before any stream
 * capture. The address is kept for the life of the process: after cudaDeviceReset on a
 * device (which also invalidates every model and buffer on it), this entry point must not be
 * called on that device again in the same process. All calls share the array and each clears
 * the keys it uses, so calls whose work overlaps on the GPU race: issue them on one stream. */
#define QW_NOALLOC_MAX_ROWS 8
qw_status qw_lm_head_argmax_noalloc(const qw_model* m, int B, const float* dev_x, float* dev_logits,
                                    int32_t* dev_next_ids, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QW_H */
