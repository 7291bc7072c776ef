/*
 * tfm.h - C ABI of libtfm, a GB300 (sm_103a) forward pass of a pre-norm
 * decoder-only Transformer language model.
 *
 * The model is the one the CS336 Transformer walkthrough assembles
 * ("手把手带工程同学从零实现一个完整的 LLM（CS336）——Transformer 篇",
 * dujian.net, section 5.7 组装 Transformer) and that "LLM 2: Transformer
 * 原理与实现" (juejin.cn) writes as h' = h + Attn(Norm(h)),
 * h_next = h' + FFN(Norm(h')):
 *
 *   h = E[tokens]
 *   for each layer:  h += Wo . Attn(RoPE(Wq u), RoPE(Wk u), Wv u),  u = RMSNorm(h) * g1
 *                    h += W2 . (silu(W1 u) * W3 u),                  u = RMSNorm(h) * g2
 *   logits = Wlm . (RMSNorm(h) * gf)
 *
 * with bias-free linears stored (out_features, in_features) row-major, RoPE on
 * adjacent coordinate pairs, causal softmax attention scaled by 1/sqrt(d_head)
 * and grouped-query heads (query head h reads kv head h / (n_head / n_kv_head)).
 *
 * Conventions for every function below:
 *  - Pointers are plain addresses.  "device" pointers must be CUDA device (or
 *    managed) memory of the current device; "host" pointers are host memory
 *    (page-locked for asynchronous copies).  The caller owns every buffer it
 *    passes; the library keeps no pointer to a caller buffer after a call
 *    returns (tfm_load_weights copies the weights into the handle's own
 *    storage).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Compute calls enqueue work on that stream and return without
 *    synchronising, allocating or freeing memory, except where a function's
 *    comment names a first call that does: tfm_forward_loss sizing its scratch,
 *    tfm_forward_graph, tfm_forward_host_async and tfm_decode_step recording a
 *    CUDA graph.
 *  - Every function returns a tfm_status.  Argument errors are found on the
 *    host before anything is launched (TFM_EINVAL / TFM_EUNSUPPORTED) and
 *    leave outputs untouched.  Errors found on the device (a token id outside
 *    [0, vocab), a pipeline wait that gave up) set a sticky device error word
 *    that tfm_device_status() reads and clears.  tfm_last_error() gives a
 *    thread-local message for the last failing call.
 *  - "bf16 mode" stores weights and activations in bfloat16 and accumulates in
 *    fp32 (tcgen05 tensor cores); the residual stream and logits are fp32.
 *    "fp32 mode" keeps everything in fp32 (CUDA-core FFMA).
 */
#ifndef TFM_H
#define TFM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TFM_OK = 0,
    TFM_EINVAL = 1,        /* bad argument: shape, pointer, alignment, mode */
    TFM_ENOMEM = 2,        /* device allocation failed (tfm_create / tfm_load_weights only) */
    TFM_ECUDA = 3,         /* a CUDA runtime call failed; see tfm_last_error() */
    TFM_EBADTOKEN = 4,     /* device: a token id was outside [0, vocab); its row was zeroed */
    TFM_ETIMEOUT = 5,      /* device: a bounded pipeline wait gave up; outputs are invalid */
    TFM_EUNSUPPORTED = 6   /* valid request the library does not implement (e.g. d_head 48 in bf16) */
} tfm_status;

typedef enum { TFM_FP32 = 0, TFM_BF16 = 1 } tfm_mode;

/* Model hyper-parameters.  Mirrors the TransformerLM constructor of the CS336
 * walkthrough, section 5.7 (vocab_size, num_layers, d_model, num_heads, d_ff,
 * theta, max_seq_len), plus n_kv_head for grouped-query attention ("LLM 2",
 * section GQA / MQA) and the batch bound that sizes the workspace.
 * Constraints (checked by tfm_validate_config):
 *   d_model % n_head == 0 (the walkthrough's assert), d_head = d_model / n_head
 *   even (RoPE pairs coordinates), n_head % n_kv_head == 0, all sizes > 0
 *   (n_layer >= 0), norm_eps > 0, rope_theta > 1.
 *   bf16 mode additionally: d_head in {32, 64, 128}, d_model % 64 == 0,
 *   d_ff % 8 == 0, vocab >= 1.  fp32 mode: d_head <= 128. */
typedef struct {
    int32_t vocab;
    int32_t d_model;
    int32_t n_head;
    int32_t n_kv_head;
    int32_t n_layer;
    int32_t d_ff;
    int32_t max_seq;
    int32_t max_batch;
    float rope_theta;
    float norm_eps;
    int32_t mode;          /* tfm_mode */
} tfm_config;

/* Weights, all row-major (out_features, in_features) like the walkthrough's
 * Linear (section 5.3).  Matrices are bf16 in bf16 mode and fp32 in fp32 mode;
 * the RMSNorm gains are always fp32.  Per-layer entries are arrays of n_layer
 * pointers.  Shapes, with Dq = n_head*d_head and Dkv = n_kv_head*d_head:
 *   embed [vocab, d_model]; attn_norm, ffn_norm, final_norm [d_model];
 *   wq [Dq, d_model]; wk, wv [Dkv, d_model]; wo [d_model, Dq];
 *   w1 (gate), w3 (up) [d_ff, d_model]; w2 (down) [d_model, d_ff];
 *   lm_head [vocab, d_model] (may be the same pointer as embed: tied weights). */
typedef struct {
    const void* embed;
    const void* const* attn_norm;
    const void* const* wq;
    const void* const* wk;
    const void* const* wv;
    const void* const* wo;
    const void* const* ffn_norm;
    const void* const* w1;
    const void* const* w3;
    const void* const* w2;
    const void* final_norm;
    const void* lm_head;
} tfm_weights;

/* ABI version of this header; bumps on any incompatible change. */
int32_t tfm_abi_version(void);

/* Host only, touches no GPU: checks a config against the constraints above. */
tfm_status tfm_validate_config(const tfm_config* cfg);

/* Host only: bytes of device workspace tfm_create allocates for cfg
 * (activations for max_batch x max_seq tokens, the RoPE table and the
 * forward_host staging buffers), 0 if the config is invalid. */
size_t tfm_workspace_bytes(const tfm_config* cfg);

/* Host only: bytes of packed weights tfm_load_weights keeps on the device. */
size_t tfm_weight_bytes(const tfm_config* cfg);

/* Creates a model handle on the current device: validates cfg, allocates the
 * workspace and the packed-weight storage, builds the RoPE cos/sin table in
 * float64 on the host (angle = position * theta^(-2i/d_head), "LLM 2",
 * section RoPE) and uploads it as fp32.  Blocking.  *handle is set only on
 * TFM_OK; release it with tfm_destroy. */
tfm_status tfm_create(const tfm_config* cfg, void** handle);

/* Copies the weights into the handle's own storage, packing [Wq; Wk; Wv] into
 * one (Dq + 2 Dkv, d_model) matrix.  weights_on_host = 1: the pointers are
 * host memory; 0: device memory.  Blocking; the caller may free its copies
 * afterwards. */
tfm_status tfm_load_weights(void* handle, const tfm_weights* w, int32_t weights_on_host);

/* ---- GPT-2-style family (a second model the pages build): absolute
 * positions added to the token embedding (a learned table, "从零构建大语言模型"
 * section 3.2 and the CS336 walkthrough's TinyGPT; or the sinusoidal table,
 * "Chapter 4: Implement a Transformer from Scratch" section 2), LayerNorm with
 * gain and shift, biased linears, a fused qkv projection, an MLP
 * fc2(GELU(fc(x))) with the exact GELU (Chapter 4 section 4; CS336 walkthrough
 * (fengye404.top) section 9 GELUFFN), no RoPE, a final LayerNorm and an LM head
 * that may be tied to the embedding and may carry a bias:
 *   h = E[tokens] + P[position]
 *   pre-norm:  h += proj(Attn(qkv(LN1(h)))),  h += fc2(GELU(fc(LN2(h))))
 *   post-norm: h = LN1(h + proj(Attn(qkv(h)))), h = LN2(h + fc2(GELU(fc(h))))
 *              (the CS336 walkthrough's pre_norm=False switch, section 10)
 *   logits = lm_head . LNf(h) (+ lm_bias)
 * tfm_config is read as for the first family except rope_theta (unused, not
 * checked); d_ff is the MLP width (4 d_model in the pages).  The forward,
 * graph, host-buffer and cross-entropy entry points take either kind of
 * handle, and so do the KV cache and decoding (a step adds the position row of
 * its position, read on the device). */
typedef enum { TFM_POS_LEARNED = 0, TFM_POS_SINUSOIDAL = 1 } tfm_pos_kind;
typedef struct {
    int32_t pos;           /* tfm_pos_kind */
    int32_t post_norm;     /* 0: pre-norm blocks; 1: post-norm blocks */
    int32_t lm_bias;       /* 1: the LM head has a bias */
} tfm_gpt2_options;

/* Weights of the GPT-2-style family.  Matrices (out_features, in_features)
 * row-major, bf16 in bf16 mode and fp32 in fp32 mode; LayerNorm gains/shifts and
 * biases fp32.  Per-layer entries are arrays of n_layer pointers.  With
 * Nqkv = (n_head + 2 n_kv_head) d_head:
 *   embed [vocab, d_model]; pos [max_seq, d_model] (learned positions; ignored
 *   for sinusoidal, which the library builds in float64 and stores in the
 *   matrix type); ln1_g, ln1_b, ln2_g, ln2_b [d_model]; w_qkv [Nqkv, d_model]
 *   (rows q | k | v), b_qkv [Nqkv]; w_proj [d_model, n_head d_head], b_proj
 *   [d_model]; w_fc [d_ff, d_model], b_fc [d_ff]; w_fc2 [d_model, d_ff], b_fc2
 *   [d_model]; lnf_g, lnf_b [d_model]; lm_head [vocab, d_model] (may be the
 *   embed pointer: tied); lm_bias [vocab] (when options.lm_bias). */
typedef struct {
    const void* embed;
    const void* pos;
    const void* const* ln1_g;
    const void* const* ln1_b;
    const void* const* w_qkv;
    const void* const* b_qkv;
    const void* const* w_proj;
    const void* const* b_proj;
    const void* const* ln2_g;
    const void* const* ln2_b;
    const void* const* w_fc;
    const void* const* b_fc;
    const void* const* w_fc2;
    const void* const* b_fc2;
    const void* lnf_g;
    const void* lnf_b;
    const void* lm_head;
    const void* lm_bias;
} tfm_gpt2_weights;

/* As tfm_create, for the GPT-2-style family with the given options.  Errors:
 * TFM_EINVAL for a NULL opt, an unknown position kind, an odd d_model or the
 * tfm_create checks (rope_theta excepted). */
tfm_status tfm_create_gpt2(const tfm_config* cfg, const tfm_gpt2_options* opt, void** handle);

/* As tfm_load_weights, for a tfm_create_gpt2 handle (TFM_EINVAL otherwise, and
 * tfm_load_weights refuses a GPT-2-style handle). */
tfm_status tfm_load_gpt2_weights(void* handle, const tfm_gpt2_weights* w, int32_t weights_on_host);

/* Forward pass of the CS336 walkthrough's TransformerLM.forward (section 5.7):
 * tokens [B, S] int32 (device) -> logits [B*S, ld_logits] fp32 (device), row
 * b*S + s holding the vocab scores of token s of sequence b in columns
 * [0, vocab); columns [vocab, ld_logits) are not written.  Positions are
 * 0..S-1 in every sequence.  Requires 1 <= B <= max_batch, 1 <= S <= max_seq,
 * ld_logits >= vocab, ld_logits % 4 == 0, logits 16-byte aligned, tokens
 * 4-byte aligned.  Launches
 * 2 + 7 n_layer kernels on `stream`; capturable in a CUDA graph.  Calls on the
 * same handle must not overlap (they share the workspace). */
tfm_status tfm_forward(void* handle, const int32_t* tokens, int32_t B, int32_t S,
                       float* logits, int64_t ld_logits, void* stream);

/* Next-token cross-entropy of the forward over tokens [B, S] against targets
 * [B, S] (int32, device; position b*S + s is scored against targets[b*S + s],
 * normally the token after it), without writing the [B*S, vocab] logits:
 * for each position i with logits z_i, lse_i = log sum_j exp(z_i[j]) and
 * loss_i = lse_i - z_i[targets_i] ("LLM 2", section Optimize / Loss; CS336
 * walkthrough (fengye404.top), section 12 训练).  In bf16 mode the LM head's
 * GEMM keeps per row a running maximum and sum of exponentials over each tile
 * of vocab columns and the target column's logit, and a second pass merges the
 * tiles; fp32 mode materialises the logits in scratch and reduces each row.
 * Outputs (device, each may be NULL): loss [B*S] and lse [B*S] fp32,
 * mean_loss one fp32 value, the mean of loss over the B*S positions (summed in
 * a fixed order, so repeated calls agree bit for bit); targets and the
 * outputs 4-byte aligned.  Same limits as tfm_forward.  A target outside [0, vocab) gives that position a NaN loss and
 * raises TFM_EBADTOKEN in the device error word (tfm_device_status).  The
 * first call for a larger B*S allocates the scratch (blocking); later calls
 * launch 3 + 7 n_layer kernels (4 + 7 n_layer with mean_loss) on `stream`.
 * Calls on the same handle must not overlap. */
tfm_status tfm_forward_loss(void* handle, const int32_t* tokens, const int32_t* targets, int32_t B,
                            int32_t S, float* loss, float* lse, float* mean_loss, void* stream);

/* Sliding-window attention per layer (hybrid models: "LLM 2", section
 * 滑动窗口和混合注意力 — most layers local, a few full): windows[l] >= 0 is layer
 * l's window (query i sees keys i - w < j <= i; 0 = full causal attention), n
 * = n_layer, or n = 0 to make every layer full again.  Applies to every later
 * forward, loss and decode call of the handle (a decode step then reads only
 * the window's positions of the cache); recorded forwards and decode steps are
 * dropped and recorded again.  Windowed layers run the same persistent
 * tensor-core attention kernels with the band's tile skip (key tiles wholly
 * before a query tile's window are never loaded).
 * Host only, not stream-ordered: call it between forwards.  TFM_EINVAL for
 * n not in {0, n_layer} or a negative window. */
tfm_status tfm_set_attention_windows(void* handle, const int32_t* windows, int32_t n);

/* tfm_forward replayed from a CUDA graph.  The first call for a given
 * (tokens, B, S, logits, ld_logits, stream) records the launch sequence into a
 * graph (nothing executes while recording), instantiates it and launches it;
 * later calls with the same arguments only launch the graph, which removes the
 * per-kernel host launch cost.  Other arguments record another graph (the four
 * most recently used recordings are kept).  Same results and
 * requirements as tfm_forward; `stream` must not be the legacy default stream
 * (NULL); per-kernel profiling does not apply to graph launches. */
tfm_status tfm_forward_graph(void* handle, const int32_t* tokens, int32_t B, int32_t S,
                             float* logits, int64_t ld_logits, void* stream);

/* The same forward with HOST buffers: copies tokens host->device, runs the
 * forward, copies logits device->host, all enqueued on `stream` (the caller
 * synchronises).  tokens_host [B, S]; logits_host [B*S, ld_logits].  When
 * ld_logits == round_up(vocab, 4) the rows are copied as one block and columns
 * [vocab, ld_logits) receive zeros; otherwise only columns [0, vocab) are
 * written. */
tfm_status tfm_forward_host(void* handle, const int32_t* tokens_host, int32_t B, int32_t S,
                            float* logits_host, int64_t ld_logits, void* stream);

/* Host round trip with the logits copy overlapped: copies tokens host->device
 * and runs the forward (replayed from a recorded graph, as tfm_forward_graph) on
 * `stream`, into one of two device logits buffers of the handle taken in turn;
 * the device->host copy of the logits then runs on the handle's own copy
 * stream, so it overlaps the next call's forward.  A buffer is written again only
 * after its previous copy has completed.  Returns once everything is enqueued.
 * The logits of a call are in logits_host [B*S, ld_logits] (columns [vocab,
 * ld_logits) as for tfm_forward_host) once the caller has made a stream wait
 * with tfm_forward_host_join and that
 * stream has reached the wait.  logits_host should be pinned (page-locked) for
 * the copy to be asynchronous; tokens_host may be reused as soon as `stream`
 * has passed the call.  Same requirements as tfm_forward_graph otherwise
 * (`stream` must not be NULL). */
tfm_status tfm_forward_host_async(void* handle, const int32_t* tokens_host, int32_t B, int32_t S,
                                  float* logits_host, int64_t ld_logits, void* stream);

/* Makes `stream` wait (without blocking the host) for every logits copy that
 * tfm_forward_host_async has issued on this handle so far. */
tfm_status tfm_forward_host_join(void* handle, void* stream);

/* ---- Incremental decoding with a KV cache ("LLM 2", sections KV cache and
 * GQA / MQA: keys and values of the positions already seen are kept, a new token
 * computes only its own q, k, v).  bf16 mode; d_head in {32, 64, 128}; H / Hkv in
 * {1, 2, 4, 8, 16} (at most 8 for d_head 128). */

/* Allocates the handle's cache once: per layer K and V, [max_batch, n_kv_head,
 * max_seq, d_head] bf16 (2 * n_layer * max_batch * n_kv_head * max_seq * d_head
 * * 2 bytes), plus the decode attention's scratch.  TFM_ENOMEM if it does not
 * fit, TFM_EUNSUPPORTED outside the shapes above.  Freed by tfm_destroy. */
tfm_status tfm_kv_cache_create(void* handle);

/* tfm_forward (same arguments and results) that also stores every layer's k
 * (after RoPE) and v of positions [0, S) of sequences [0, B) in the cache; the
 * cache then holds S positions for B sequences. */
tfm_status tfm_prefill(void* handle, const int32_t* tokens, int32_t B, int32_t S, float* logits,
                       int64_t ld_logits, void* stream);

/* One new token per sequence: tokens [B] (device) at position pos, which must be
 * the cached length (pos < max_seq; B the prefill's batch).  Appends its k, v to
 * every layer's cache and writes logits [B, ld_logits] (row b: the scores of the
 * next token after position pos of sequence b, columns [0, vocab)), the same as
 * row pos of tfm_forward over the sequence extended by this token.  The cached
 * length becomes pos + 1.  Calls on a handle are ordered on the host in the order
 * they are made (the length is advanced at enqueue time).  A step whose B,
 * logits, ld_logits and stream equal the previous step's is recorded into a
 * CUDA graph (the position and tokens are read on the device, so the recording
 * serves every later position) and replayed from then on; the two most recent
 * recordings are kept.  Steps on the legacy default stream (NULL) or with
 * profiling on launch their kernels directly. */
tfm_status tfm_decode_step(void* handle, const int32_t* tokens, int32_t B, int32_t pos,
                           float* logits, int64_t ld_logits, void* stream);

/* Synchronises the device, then returns and clears the sticky device error word
 * (TFM_OK, TFM_EBADTOKEN or TFM_ETIMEOUT), or TFM_ECUDA if the context faulted.
 * handle may be NULL (component calls share the same word). */
tfm_status tfm_device_status(void* handle);

/* Self-test of the failure-detection path: launches one small kernel that waits
 * on an mbarrier nothing will ever complete, with the same bounded-wait code as
 * the pipelines but a limit of `limit_ms` milliseconds (1..2000).  The wait gives
 * up, the kernel latches TFM_ETIMEOUT in the device error word and returns, so
 * a following tfm_device_status() returns TFM_ETIMEOUT and the context stays
 * usable.  No fault, trap or hang is involved. */
tfm_status tfm_selftest_wait_timeout(int32_t limit_ms, void* stream);

/* Thread-local text of the last error raised on this thread ("" if none). */
const char* tfm_last_error(void);

/* Frees everything the handle owns.  NULL is a no-op. */
void tfm_destroy(void* handle);

/* ---------------------------------------------------------------- profiling
 * Per-kernel CUDA-event timing of tfm_forward.  While enabled, every forward
 * records an event on its stream before the first launch and after each
 * launch (cheap stream operations; not capturable in a CUDA graph).
 * tfm_profile_read() synchronises those events and adds, per kernel kind, the
 * elapsed milliseconds and launch counts of every forward since the last read
 * into ms[kind] and launches[kind] (arrays of TFM_PROFILE_KINDS entries, which
 * the caller zeroes), then forgets them.  Kinds: 0 embedding fused with the
 * first RMSNorm, 1 RMSNorm,
 * 2 QKV projection + RoPE, 3 attention, 4 output projection + residual,
 * 5 gate/up projection + SwiGLU, 6 down projection + residual, 7 LM head. */
#define TFM_PROFILE_KINDS 8
tfm_status tfm_profile_enable(void* handle, int32_t enable);
tfm_status tfm_profile_read(void* handle, double* ms, int64_t* launches);
const char* tfm_profile_kind_name(int32_t kind);

/* ---------------------------------------------------------------- components
 * Single operations on caller buffers (device pointers), for testing each step
 * against the oracle and for callers that assemble their own model.
 * Empty calls (M = 0; B, H or S = 0 for RoPE; B or S = 0 for attention; B = 0
 * for decode attention) check their other arguments, then return TFM_OK
 * without launching anything or reading any pointer, which may then be NULL. */

/* Embedding lookup (CS336 walkthrough, section 5.2): h[m, :] = E[tokens[m], :]
 * as fp32.  tokens [M] int32; E [V, D] bf16 or fp32 (mode); h [M, D] fp32.
 * An id outside [0, V) writes a zero row and sets TFM_EBADTOKEN.  E and h
 * 16-byte aligned, tokens 4-byte aligned, else TFM_EINVAL. */
tfm_status tfm_embedding(const int32_t* tokens, const void* E, float* h, int64_t M,
                         int32_t V, int32_t D, int32_t mode, void* stream);

/* RMSNorm (CS336 walkthrough, section 5.6): y = x / sqrt(mean(x^2) + eps) * g
 * per row, computed in fp32 and rounded once at the end.  x [M, D] fp32,
 * g [D] fp32, y [M, D] bf16 (out_mode TFM_BF16) or fp32 (TFM_FP32).
 * D % 8 == 0 and 16-byte aligned pointers are required. */
tfm_status tfm_rmsnorm(const float* x, const float* g, void* y, int64_t M, int32_t D,
                       float eps, int32_t out_mode, void* stream);

/* RoPE in place (CS336 walkthrough, section 5.5; "LLM 2", section RoPE):
 * x [B, H, S, dh] (bf16 or fp32), each adjacent pair (x[2i], x[2i+1]) of token
 * s turned by pos * theta^(-2i/dh), pos = positions[b*S + s] (int32 [B, S],
 * device) or s when positions is NULL.  dh even, dh <= 256.  x aligned to its
 * element size and positions to 4 bytes, else TFM_EINVAL. */
tfm_status tfm_rope(void* x, const int32_t* positions, int32_t B, int32_t H, int32_t S,
                    int32_t dh, float theta, int32_t mode, void* stream);

/* Causal scaled dot-product attention (CS336 walkthrough, section 5.4):
 * o = softmax(q k^T * scale + M) v with M = -inf above the diagonal, per
 * sequence and head; query head h reads kv head h / (H / Hkv) ("LLM 2",
 * section GQA / MQA).  q [B, H, S, dh]; k, v [B, Hkv, S, dh]; o [B, S, H*dh]
 * (heads merged back, the layout the output projection reads).  scale <= 0
 * means 1/sqrt(dh).  bf16 mode: dh in {32, 64, 128}; fp32 mode: dh <= 128. */
tfm_status tfm_causal_attention(const void* q, const void* k, const void* v, void* o,
                                int32_t B, int32_t H, int32_t Hkv, int32_t S, int32_t dh,
                                float scale, int32_t mode, void* stream);

/* tfm_causal_attention with a sliding window ("LLM 2", section
 * 滑动窗口和混合注意力: each token sees a local band of the causal graph):
 * query i attends to keys j with i - window < j <= i (itself and the
 * window - 1 positions before it); window = 0, or window >= S, is plain causal
 * attention.  Key tiles entirely before a query tile's window are never loaded.
 * TFM_EINVAL for window < 0; otherwise as tfm_causal_attention. */
tfm_status tfm_causal_attention_window(const void* q, const void* k, const void* v, void* o,
                                       int32_t B, int32_t H, int32_t Hkv, int32_t S, int32_t dh,
                                       float scale, int32_t window, int32_t mode, void* stream);

/* Attention of one new query per sequence over a KV cache, the attention of a
 * decode step ("LLM 2", sections KV cache and GQA / MQA; the last row of the
 * causal mask of the CS336 walkthrough, section 5.4): q [B, H, dh] (the query of
 * position pos), k_cache and v_cache [B, Hkv, max_seq, dh] holding positions
 * [0, pos], o [B, H*dh]; o = softmax(q k^T * scale) v over positions
 * [max(0, pos - window + 1), pos] (window 0: all of [0, pos]), query head h
 * reading kv head h / (H / Hkv); scale <= 0 means 1/sqrt(dh).  bf16 only;
 * dh in {32, 64, 128}; H / Hkv in {1, 2, 4, 8, 16} (<= 8 at dh 128).  The keys
 * are split over CTAs in chunks of 8192/dh positions, each fetched by bulk
 * asynchronous copies, and the chunks are merged exactly by a second kernel.
 * workspace: device, 16-byte aligned, at least
 * tfm_decode_attention_workspace_bytes(B, H, max_seq, dh) bytes, not used by
 * another call in flight.  The position goes to the workspace by a small
 * host-to-device copy on `stream`, so the call cannot be recorded into a graph:
 * on a capturing stream it returns TFM_EINVAL before enqueueing anything
 * (tfm_decode_step can be recorded).  TFM_EINVAL for bad sizes (0 <= pos < max_seq,
 * window >= 0) or a small workspace; TFM_EUNSUPPORTED for other dh / groups. */
size_t tfm_decode_attention_workspace_bytes(int32_t B, int32_t H, int32_t max_seq, int32_t dh);
tfm_status tfm_decode_attention(const void* q, const void* k_cache, const void* v_cache, void* o,
                                int32_t B, int32_t H, int32_t Hkv, int32_t max_seq, int32_t pos,
                                int32_t dh, float scale, int32_t window, void* workspace,
                                size_t workspace_bytes, void* stream);

/* Bias-free Linear (CS336 walkthrough, section 5.3): y = x W^T.
 * x [M, K], W [N, K] (bf16 or fp32 by mode); y [M, ldy] fp32 when
 * out_fp32 != 0 (accumulate != 0 adds into y instead of overwriting), else
 * bf16 [M, ldy] (bf16 mode only; accumulate must be 0).  K % 8 == 0 in bf16
 * mode; ldy >= N, ldy % 8 == 0. */
tfm_status tfm_linear(const void* x, const void* W, void* y, int64_t M, int32_t N, int32_t K,
                      int64_t ldy, int32_t out_fp32, int32_t accumulate, int32_t mode,
                      void* stream);

/* SwiGLU feed-forward (CS336 walkthrough, section 5.3):
 * y (+)= W2 (silu(W1 x) * W3 x), silu(z) = z / (1 + exp(-z)).
 * x [M, D], w1 and w3 [F, D], w2 [D, F] (bf16 or fp32 by mode); y [M, D] fp32,
 * overwritten (accumulate 0) or added to (accumulate 1, the residual add).
 * The hidden activation [M, F] lives in the caller's `workspace` of at least
 * tfm_swiglu_workspace_bytes(M, F, mode) bytes (device, 256-byte aligned). */
tfm_status tfm_swiglu(const void* x, const void* w1, const void* w3, const void* w2, float* y,
                      int64_t M, int32_t D, int32_t F, int32_t accumulate,
                      void* workspace, size_t workspace_bytes, int32_t mode, void* stream);
size_t tfm_swiglu_workspace_bytes(int64_t M, int32_t F, int32_t mode);

/* tfm_swiglu for callers that cannot allocate device memory.  The tutorial
 * pages have no counterpart: this is a deployment convenience of the library.
 *
 * Who needs it: plugins running inside a host framework that owns the device
 * allocator (and may have given all free memory to its own pool), and
 * deployments whose device memory is budgeted once at start-up, where a later
 * cudaMalloc would fail or break the budget.  Arguments and results are those of
 * tfm_swiglu without the workspace: the [M, F] hidden activation lives in a
 * fixed array the library declares in device memory, of
 * tfm_swiglu_noalloc_max_bytes() bytes (16 MiB) per device, held on every GPU
 * that loads the library until the process exits.  A call whose activation
 * (tfm_swiglu_workspace_bytes(M, F, mode)) does not fit, or M < 0 or F < 1,
 * returns TFM_EINVAL.
 * No allocator is called, not even on the first call; that first call on each
 * device looks up the array's device address (cudaGetSymbolAddress) with that
 * device current.
 * All calls share the array and it keeps the last call's contents
 * (nothing needs clearing: each call overwrites every entry it reads); calls
 * whose kernels overlap on the GPU race on it, so order them on one stream. */
tfm_status tfm_swiglu_noalloc(const void* x, const void* w1, const void* w3, const void* w2,
                              float* y, int64_t M, int32_t D, int32_t F, int32_t accumulate,
                              int32_t mode, void* stream);
size_t tfm_swiglu_noalloc_max_bytes(void);

#ifdef __cplusplus
}
#endif
#endif /* TFM_H */
