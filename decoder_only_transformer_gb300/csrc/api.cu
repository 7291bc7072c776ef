// api.cu - host side of the libtfm C ABI (include/tfm.h): argument checks,
// the model handle (workspace, packed weights, RoPE table), the forward
// launch sequence and the single-operation entry points.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

// Sticky device error word (one per device; see tfm_device_status).
__device__ int g_tfm_err_word;

namespace tfm {

namespace {

thread_local std::string t_last_error;

tfm_status fail(tfm_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return s;
}

tfm_status cuda_fail(cudaError_t e, const char* what) {
    return fail(TFM_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
int* g_err_addr[kMaxDevices];
int g_sms[kMaxDevices];

int current_device() {
    int d = 0;
    cudaGetDevice(&d);
    return (d >= 0 && d < kMaxDevices) ? d : 0;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Element alignment of a typed array (n a power of two); kernels read int32 ids
// and fp32 scalars with naturally aligned loads.
bool aligned_to(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

}  // namespace

int* device_error_word() {
    const int d = current_device();
    std::lock_guard<std::mutex> lk(g_dev_mutex);
    if (!g_err_addr[d]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_tfm_err_word) != cudaSuccess) return nullptr;
        g_err_addr[d] = static_cast<int*>(p);
    }
    return g_err_addr[d];
}

int sm_count() {
    const int d = current_device();
    std::lock_guard<std::mutex> lk(g_dev_mutex);
    if (!g_sms[d]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0)
            n = 148;
        g_sms[d] = n;
    }
    return g_sms[d];
}

const char* cuda_error_text(cudaError_t e) { return cudaGetErrorString(e); }

void set_last_error(const char* msg) { t_last_error = msg ? msg : ""; }

// ------------------------------------------------------------------ config
namespace {

tfm_status check_config(const tfm_config* c, int arch = 0) {
    if (!c) return fail(TFM_EINVAL, "config is NULL");
    if (c->vocab < 1 || c->d_model < 1 || c->n_head < 1 || c->n_kv_head < 1 || c->n_layer < 0 ||
        c->d_ff < 1 || c->max_seq < 1 || c->max_batch < 1)
        return fail(TFM_EINVAL, "sizes must be positive (n_layer >= 0)");
    if (c->mode != TFM_FP32 && c->mode != TFM_BF16) return fail(TFM_EINVAL, "unknown mode %d", c->mode);
    if (c->d_model % c->n_head) return fail(TFM_EINVAL, "d_model %% n_head != 0");
    if (c->n_head % c->n_kv_head) return fail(TFM_EINVAL, "n_head %% n_kv_head != 0");
    const int dh = c->d_model / c->n_head;
    if (dh % 2) return fail(TFM_EINVAL, "d_head must be even for RoPE");
    if (!(c->norm_eps > 0.f) || !std::isfinite(c->norm_eps)) return fail(TFM_EINVAL, "norm_eps must be > 0");
    if (arch == 0 && (!(c->rope_theta > 1.f) || !std::isfinite(c->rope_theta)))
        return fail(TFM_EINVAL, "rope_theta must be > 1");
    if ((int64_t)c->max_seq * c->max_batch > (int64_t)1 << 30) return fail(TFM_EINVAL, "max_batch*max_seq too large");
    if (c->mode == TFM_BF16) {
        if (dh != 32 && dh != 64 && dh != 128)
            return fail(TFM_EUNSUPPORTED, "bf16 mode supports d_head 32, 64, 128 (got %d)", dh);
        if (c->d_model % 64) return fail(TFM_EUNSUPPORTED, "bf16 mode needs d_model %% 64 == 0");
        if (c->d_ff % 8) return fail(TFM_EUNSUPPORTED, "bf16 mode needs d_ff %% 8 == 0");
    } else {
        if (dh % 8 || dh > 128) return fail(TFM_EUNSUPPORTED, "fp32 mode needs d_head %% 8 == 0, <= 128");
        if (c->d_model % 8) return fail(TFM_EUNSUPPORTED, "fp32 mode needs d_model %% 8 == 0");
        if (c->d_ff % 4) return fail(TFM_EUNSUPPORTED, "fp32 mode needs d_ff %% 4 == 0");
    }
    return TFM_OK;
}

inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// float -> bf16 bit pattern, round to nearest, ties to even (finite values).
inline uint16_t bf16_bits_rne(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

struct Sizes {
    int64_t M, D, Dq, Dkv, Nqkv, F, V, ldV, es;   // es = element size of matrices/activations
};

Sizes sizes_of(const tfm_config* c) {
    Sizes s;
    s.M = (int64_t)c->max_batch * c->max_seq;
    s.D = c->d_model;
    const int64_t dh = c->d_model / c->n_head;
    s.Dq = c->n_head * dh;
    s.Dkv = c->n_kv_head * dh;
    s.Nqkv = s.Dq + 2 * s.Dkv;
    s.F = c->d_ff;
    s.V = c->vocab;
    s.ldV = round_up(s.V, 4);
    s.es = c->mode == TFM_BF16 ? 2 : 4;
    return s;
}

// Workspace carve-up, every piece 256-byte aligned.
struct Layout {
    size_t h, xn, q, k, v, o, a, rope, tok, logits, logits2, total;
};

Layout layout_of(const tfm_config* c) {
    const Sizes s = sizes_of(c);
    Layout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += (bytes + 255) / 256 * 256;
        return at;
    };
    const int64_t dh = c->d_model / c->n_head;
    L.h = take(s.M * s.D * 4);
    L.xn = take(s.M * s.D * s.es);
    L.q = take(s.M * s.Dq * s.es);
    L.k = take(s.M * s.Dkv * s.es);
    L.v = take(s.M * s.Dkv * s.es);
    L.o = take(s.M * s.Dq * s.es);
    L.a = take(s.M * s.F * s.es);
    L.rope = take((size_t)c->max_seq * (dh / 2) * 8);
    L.tok = take(s.M * 4);
    L.logits = take(s.M * s.ldV * 4);
    L.logits2 = take(s.M * s.ldV * 4);    // second buffer of tfm_forward_host_async
    L.total = off;
    return L;
}

size_t weight_bytes_of(const tfm_config* c) {
    const Sizes s = sizes_of(c);
    // matrices and gains of one layer (9 pieces), plus embed, final_norm and
    // lm_head; each piece is rounded up to 256 bytes by the loader.
    const size_t per_layer =
        (size_t)(s.Nqkv * s.D + s.D * s.Dq + 2 * s.F * s.D + s.D * s.F) * s.es + 2 * s.D * 4;
    return (size_t)c->n_layer * (per_layer + 9 * 256) + 2 * (size_t)s.V * s.D * s.es + s.D * 4 +
           3 * 256;
}

// GPT-2-style family: matrices (fused qkv, proj, fc, fc2), LayerNorm gains and
// shifts, biases per layer; embed, position table, final LayerNorm, LM head and
// its bias; each piece rounded up to 256 bytes.
size_t gpt2_weight_bytes_of(const tfm_config* c) {
    const Sizes s = sizes_of(c);
    const size_t per_layer =
        (size_t)(s.Nqkv * s.D + s.D * s.Dq + 2 * s.F * s.D) * s.es +
        (size_t)(4 * s.D + s.Nqkv + s.D + s.F + s.D) * 4;
    return (size_t)c->n_layer * (per_layer + 12 * 256) + 2 * (size_t)s.V * s.D * s.es +
           (size_t)c->max_seq * s.D * s.es + 2 * s.D * 4 + s.V * 4 + 6 * 256;
}

}  // namespace

// ------------------------------------------------------------------ handle
struct Model {
    tfm_config cfg;
    Sizes sz;
    Layout lay;
    int device = 0;
    uint8_t* ws = nullptr;         // workspace
    uint8_t* wmem = nullptr;       // packed weights
    size_t wbytes = 0;
    bool loaded = false;
    // packed weights (device pointers into wmem)
    void* embed = nullptr;
    void* lm_head = nullptr;
    float* final_norm = nullptr;
    std::vector<float*> attn_norm, ffn_norm;
    std::vector<void*> wqkv, wo, w1, w3, w2;
    // GPT-2-style family (tfm_create_gpt2): attn_norm / ffn_norm / final_norm
    // hold the LayerNorm gains, wqkv the fused qkv, wo the projection, w1 / w2
    // the MLP's fc / fc2; these hold the rest
    int arch = 0;                   // 0: RMSNorm / RoPE / SwiGLU; 1: GPT-2-style
    tfm_gpt2_options g2{};
    void* pos = nullptr;            // position rows [max_seq, D], matrix type
    std::vector<float*> ln1_b, ln2_b, b_qkv, b_proj, b_fc, b_fc2;
    float* lnf_b = nullptr;
    float* lm_bias = nullptr;
    // sliding window of each layer's attention (tfm_set_attention_windows; 0: full)
    std::vector<int> windows;
    // cached tensor-core plans for the current token count
    int64_t plan_m = -1;
    std::vector<GemmPlan> p_qkv, p_o, p_gu, p_down;
    GemmPlan p_lm;
    AttnPlan p_attn;               // tcgen05 attention
    const float* plan_logits = nullptr;
    int64_t plan_ld = -1;
    int plan_S = -1;
    // recorded forwards (tfm_forward_graph, tfm_forward_host_async) and the
    // arguments each was recorded for; a few are kept, least recently used out
    struct Graph {
        cudaGraphExec_t exec = nullptr;
        const void* tokens = nullptr;
        const float* logits = nullptr;
        int B = 0, S = 0;
        int64_t ld = 0;
        void* stream = nullptr;
        uint64_t used = 0;
    };
    static constexpr int kGraphs = 4;
    Graph graphs[kGraphs];
    uint64_t graph_clock = 0;
    // KV cache (tfm_kv_cache_create): per layer K then V, each [max_batch, Hkv,
    // max_seq, dh]; decode attention scratch; filled positions and batch
    uint8_t* kv = nullptr;
    size_t kv_layer_bytes = 0;      // one of K or V of one layer
    float* dec_part = nullptr;
    // fused cross-entropy (tfm_forward_loss): per-row LSE slots [M][slots] float2,
    // target logits [M], per-row losses [M]; fp32 mode also materialises logits
    uint8_t* loss_mem = nullptr;
    int64_t loss_rows = 0;          // rows the scratch holds
    float2* lse_part = nullptr;
    float* lse_tgt = nullptr;
    float* loss_tmp = nullptr;
    float* loss_logits = nullptr;   // fp32 mode [M, ldV]
    GemmPlan p_lse;                 // LM head with the EPI_LSE epilogue
    int lse_M = -1;
    const int32_t* lse_targets = nullptr;
    int* pos_dev = nullptr;         // position of the decode step being run (device word)
    int32_t* tok_dev = nullptr;     // its tokens [max_batch]
    Graph dgraphs[2];               // recorded decode steps (position, tokens read on the device)
    Graph dlast;                    // arguments of the previous decode step
    int kv_len = 0, kv_batch = 0;
    // tensor-core plans of a decode step (M = batch rows), cached by batch and logits
    std::vector<GemmPlan> d_qkv, d_o, d_gu, d_down;
    GemmPlan d_lm;
    int dplan_B = -1;
    // the decode GEMMs behind RMSNorms (QKV of layers after the first, gate/up,
    // LM head) compute those norms themselves (GemmPlan::norm_x)
    bool dnorm_fused = false;
    const float* dplan_logits = nullptr;
    int64_t dplan_ld = -1;
    // tfm_forward_host_async: copy stream, per-buffer events, calls so far
    cudaStream_t copy_st = nullptr;
    cudaEvent_t fwd_done[2] = {nullptr, nullptr}, copied[2] = {nullptr, nullptr};
    bool copy_pending[2] = {false, false};
    int64_t async_calls = 0;
    // per-kernel event timing (tfm_profile_*)
    bool prof = false;
    struct ProfRun {
        size_t ev0;
        std::vector<int> kinds;
    };
    std::vector<cudaEvent_t> ev_pool;
    size_t ev_used = 0;
    std::vector<ProfRun> runs;

    cudaEvent_t next_event() {
        if (ev_used == ev_pool.size()) {
            cudaEvent_t e = nullptr;
            if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
            ev_pool.push_back(e);
        }
        return ev_pool[ev_used++];
    }

    float* h() { return reinterpret_cast<float*>(ws + lay.h); }
    void* xn() { return ws + lay.xn; }
    void* q() { return ws + lay.q; }
    void* k() { return ws + lay.k; }
    void* v() { return ws + lay.v; }
    void* o() { return ws + lay.o; }
    void* a() { return ws + lay.a; }
    float* rope() { return reinterpret_cast<float*>(ws + lay.rope); }
    int32_t* tok() { return reinterpret_cast<int32_t*>(ws + lay.tok); }
    float* logits() { return reinterpret_cast<float*>(ws + lay.logits); }
    float* logits_buf(int b) { return reinterpret_cast<float*>(ws + (b ? lay.logits2 : lay.logits)); }
    void* kcache(int l) { return kv + (size_t)l * 2 * kv_layer_bytes; }
    void* vcache(int l) { return kv + ((size_t)l * 2 + 1) * kv_layer_bytes; }
};

}  // namespace tfm

using tfm::Model;
using tfm::fail;

extern "C" {

int32_t tfm_abi_version(void) { return 1; }

const char* tfm_last_error(void) { return tfm::t_last_error.c_str(); }

tfm_status tfm_validate_config(const tfm_config* cfg) { return tfm::check_config(cfg); }

size_t tfm_workspace_bytes(const tfm_config* cfg) {
    if (tfm::check_config(cfg) != TFM_OK) return 0;
    return tfm::layout_of(cfg).total;
}

size_t tfm_weight_bytes(const tfm_config* cfg) {
    if (tfm::check_config(cfg) != TFM_OK) return 0;
    return tfm::weight_bytes_of(cfg);
}

static tfm_status create_impl(const tfm_config* cfg, int arch, const tfm_gpt2_options* opt,
                              void** handle);

tfm_status tfm_create(const tfm_config* cfg, void** handle) {
    return create_impl(cfg, 0, nullptr, handle);
}

tfm_status tfm_create_gpt2(const tfm_config* cfg, const tfm_gpt2_options* opt, void** handle) {
    if (!opt) return fail(TFM_EINVAL, "NULL options");
    if (opt->pos != TFM_POS_LEARNED && opt->pos != TFM_POS_SINUSOIDAL)
        return fail(TFM_EINVAL, "unknown position kind %d", opt->pos);
    if (cfg && cfg->d_model % 2) return fail(TFM_EINVAL, "d_model must be even");
    return create_impl(cfg, 1, opt, handle);
}

static tfm_status create_impl(const tfm_config* cfg, int arch, const tfm_gpt2_options* opt,
                              void** handle) {
    if (!handle) return fail(TFM_EINVAL, "handle pointer is NULL");
    tfm_status st = tfm::check_config(cfg, arch);
    if (st != TFM_OK) return st;
    Model* m = new Model();
    m->cfg = *cfg;
    m->arch = arch;
    if (opt) m->g2 = *opt;
    m->sz = tfm::sizes_of(cfg);
    m->lay = tfm::layout_of(cfg);
    cudaGetDevice(&m->device);
    cudaError_t e = cudaMalloc(&m->ws, m->lay.total);
    if (e != cudaSuccess) {
        const size_t bytes = m->lay.total;
        delete m;
        cudaGetLastError();
        return fail(TFM_ENOMEM, "workspace of %zu bytes: %s", bytes, cudaGetErrorString(e));
    }
    m->wbytes = arch ? tfm::gpt2_weight_bytes_of(cfg) : tfm::weight_bytes_of(cfg);
    e = cudaMalloc(&m->wmem, m->wbytes);
    if (e != cudaSuccess) {
        cudaFree(m->ws);
        delete m;
        cudaGetLastError();
        return fail(TFM_ENOMEM, "weights: %s", cudaGetErrorString(e));
    }
    // RoPE table: angle = s * theta^(-2i/dh) in float64, stored as fp32
    // (cos, sin) pairs, [max_seq][dh/2][2].
    const int dh = cfg->d_model / cfg->n_head, half = dh / 2;
    std::vector<float> hcs((size_t)cfg->max_seq * half * 2);
    const double theta = arch ? 10000.0 : (double)cfg->rope_theta;   // unused by the GPT-2 family
    for (int s = 0; s < cfg->max_seq; ++s)
        for (int i = 0; i < half; ++i) {
            const double ang = (double)s * std::pow(theta, -2.0 * i / dh);
            hcs[((size_t)s * half + i) * 2] = (float)std::cos(ang);
            hcs[((size_t)s * half + i) * 2 + 1] = (float)std::sin(ang);
        }
    e = cudaMemcpy(m->rope(), hcs.data(), hcs.size() * 4, cudaMemcpyHostToDevice);
    // The internal logits buffers start zeroed: their columns [vocab, ldV) are
    // never written, so a contiguous device->host copy gives zeros there.
    if (e == cudaSuccess) e = cudaMemset(m->logits_buf(0), 0, (size_t)m->sz.M * m->sz.ldV * 4);
    if (e == cudaSuccess) e = cudaMemset(m->logits_buf(1), 0, (size_t)m->sz.M * m->sz.ldV * 4);
    if (e == cudaSuccess && !tfm::device_error_word()) e = cudaErrorSymbolNotFound;
    if (e != cudaSuccess) {
        cudaFree(m->ws);
        cudaFree(m->wmem);
        delete m;
        return tfm::cuda_fail(e, "tfm_create");
    }
    // Copy stream and events of tfm_forward_host_async (non-blocking: no implicit
    // ordering against the legacy stream).
    e = cudaStreamCreateWithFlags(&m->copy_st, cudaStreamNonBlocking);
    for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
        e = cudaEventCreateWithFlags(&m->fwd_done[b], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m->copied[b], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) {
        tfm_destroy(m);
        return tfm::cuda_fail(e, "tfm_create: copy stream");
    }
    *handle = m;
    return TFM_OK;
}

void tfm_destroy(void* handle) {
    Model* m = static_cast<Model*>(handle);
    if (!m) return;
    if (m->copy_st) cudaStreamSynchronize(m->copy_st);
    for (auto& g : m->graphs)
        if (g.exec) cudaGraphExecDestroy(g.exec);
    for (auto& g : m->dgraphs)
        if (g.exec) cudaGraphExecDestroy(g.exec);
    for (int b = 0; b < 2; ++b) {
        if (m->fwd_done[b]) cudaEventDestroy(m->fwd_done[b]);
        if (m->copied[b]) cudaEventDestroy(m->copied[b]);
    }
    if (m->copy_st) cudaStreamDestroy(m->copy_st);
    if (m->kv) cudaFree(m->kv);
    if (m->loss_mem) cudaFree(m->loss_mem);
    for (cudaEvent_t e : m->ev_pool) cudaEventDestroy(e);
    cudaFree(m->ws);
    cudaFree(m->wmem);
    delete m;
}

tfm_status tfm_load_weights(void* handle, const tfm_weights* w, int32_t weights_on_host) {
    Model* m = static_cast<Model*>(handle);
    if (!m || !w) return fail(TFM_EINVAL, "NULL handle or weights");
    if (m->arch != 0) return fail(TFM_EINVAL, "a GPT-2-style handle takes tfm_load_gpt2_weights");
    const tfm_config& c = m->cfg;
    const auto& s = m->sz;
    if (!w->embed || !w->final_norm || !w->lm_head) return fail(TFM_EINVAL, "NULL embed/final_norm/lm_head");
    if (c.n_layer > 0 && (!w->attn_norm || !w->wq || !w->wk || !w->wv || !w->wo || !w->ffn_norm ||
                          !w->w1 || !w->w3 || !w->w2))
        return fail(TFM_EINVAL, "NULL per-layer weight array");
    for (int l = 0; l < c.n_layer; ++l)
        if (!w->attn_norm[l] || !w->wq[l] || !w->wk[l] || !w->wv[l] || !w->wo[l] ||
            !w->ffn_norm[l] || !w->w1[l] || !w->w3[l] || !w->w2[l])
            return fail(TFM_EINVAL, "NULL weight pointer in layer %d", l);
    const cudaMemcpyKind kind = weights_on_host ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t* p = m->wmem + off;
        off += (bytes + 255) / 256 * 256;
        return p;
    };
    cudaError_t e = cudaSuccess;
    auto copy = [&](void* dst, const void* src, size_t bytes) {
        if (e == cudaSuccess) e = cudaMemcpy(dst, src, bytes, kind);
    };
    const size_t es = s.es;
    m->embed = take(s.V * s.D * es);
    copy(m->embed, w->embed, s.V * s.D * es);
    m->attn_norm.assign(c.n_layer, nullptr);
    m->ffn_norm.assign(c.n_layer, nullptr);
    m->wqkv.assign(c.n_layer, nullptr);
    m->wo.assign(c.n_layer, nullptr);
    m->w1.assign(c.n_layer, nullptr);
    m->w3.assign(c.n_layer, nullptr);
    m->w2.assign(c.n_layer, nullptr);
    for (int l = 0; l < c.n_layer; ++l) {
        m->attn_norm[l] = reinterpret_cast<float*>(take(s.D * 4));
        copy(m->attn_norm[l], w->attn_norm[l], s.D * 4);
        uint8_t* qkv = take(s.Nqkv * s.D * es);
        m->wqkv[l] = qkv;
        copy(qkv, w->wq[l], s.Dq * s.D * es);
        copy(qkv + s.Dq * s.D * es, w->wk[l], s.Dkv * s.D * es);
        copy(qkv + (s.Dq + s.Dkv) * s.D * es, w->wv[l], s.Dkv * s.D * es);
        m->wo[l] = take(s.D * s.Dq * es);
        copy(m->wo[l], w->wo[l], s.D * s.Dq * es);
        m->ffn_norm[l] = reinterpret_cast<float*>(take(s.D * 4));
        copy(m->ffn_norm[l], w->ffn_norm[l], s.D * 4);
        m->w1[l] = take(s.F * s.D * es);
        copy(m->w1[l], w->w1[l], s.F * s.D * es);
        m->w3[l] = take(s.F * s.D * es);
        copy(m->w3[l], w->w3[l], s.F * s.D * es);
        m->w2[l] = take(s.D * s.F * es);
        copy(m->w2[l], w->w2[l], s.D * s.F * es);
    }
    m->final_norm = reinterpret_cast<float*>(take(s.D * 4));
    copy(m->final_norm, w->final_norm, s.D * 4);
    if (w->lm_head == w->embed) {
        m->lm_head = m->embed;
    } else {
        m->lm_head = take(s.V * s.D * es);
        copy(m->lm_head, w->lm_head, s.V * s.D * es);
    }
    if (off > m->wbytes) return fail(TFM_EINVAL, "internal: weight storage overflow");
    if (e != cudaSuccess) return tfm::cuda_fail(e, "tfm_load_weights");
    m->loaded = true;
    m->plan_m = -1;
    return TFM_OK;
}

tfm_status tfm_load_gpt2_weights(void* handle, const tfm_gpt2_weights* w, int32_t weights_on_host) {
    Model* m = static_cast<Model*>(handle);
    if (!m || !w) return fail(TFM_EINVAL, "NULL handle or weights");
    if (m->arch != 1) return fail(TFM_EINVAL, "tfm_load_gpt2_weights needs a tfm_create_gpt2 handle");
    const tfm_config& c = m->cfg;
    const auto& s = m->sz;
    if (!w->embed || !w->lnf_g || !w->lnf_b || !w->lm_head)
        return fail(TFM_EINVAL, "NULL embed / lnf_g / lnf_b / lm_head");
    if (m->g2.pos == TFM_POS_LEARNED && !w->pos) return fail(TFM_EINVAL, "NULL learned position table");
    if (m->g2.lm_bias && !w->lm_bias) return fail(TFM_EINVAL, "NULL lm_bias");
    if (c.n_layer > 0 && (!w->ln1_g || !w->ln1_b || !w->w_qkv || !w->b_qkv || !w->w_proj ||
                          !w->b_proj || !w->ln2_g || !w->ln2_b || !w->w_fc || !w->b_fc ||
                          !w->w_fc2 || !w->b_fc2))
        return fail(TFM_EINVAL, "NULL per-layer weight array");
    for (int l = 0; l < c.n_layer; ++l)
        if (!w->ln1_g[l] || !w->ln1_b[l] || !w->w_qkv[l] || !w->b_qkv[l] || !w->w_proj[l] ||
            !w->b_proj[l] || !w->ln2_g[l] || !w->ln2_b[l] || !w->w_fc[l] || !w->b_fc[l] ||
            !w->w_fc2[l] || !w->b_fc2[l])
            return fail(TFM_EINVAL, "NULL weight pointer in layer %d", l);
    const cudaMemcpyKind kind = weights_on_host ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice;
    size_t off = 0;
    bool over = false;
    auto take = [&](size_t bytes) {
        uint8_t* p = m->wmem + off;
        off += (bytes + 255) / 256 * 256;
        if (off > m->wbytes) over = true;
        return p;
    };
    cudaError_t e = cudaSuccess;
    auto copy = [&](void* dst, const void* src, size_t bytes) {
        if (e == cudaSuccess && !over) e = cudaMemcpy(dst, src, bytes, kind);
    };
    const size_t es = s.es;
    m->embed = take(s.V * s.D * es);
    copy(m->embed, w->embed, s.V * s.D * es);
    m->pos = take((size_t)c.max_seq * s.D * es);
    if (m->g2.pos == TFM_POS_LEARNED) {
        copy(m->pos, w->pos, (size_t)c.max_seq * s.D * es);
    } else if (!over && e == cudaSuccess) {
        // pe[p, 2i] = sin(p / 10000^(2i/D)), pe[p, 2i+1] = cos(same), in float64,
        // stored in the matrix type ("Chapter 4", section 2 PositionalEncoding)
        std::vector<uint8_t> host((size_t)c.max_seq * s.D * es);
        for (int p = 0; p < c.max_seq; ++p)
            for (int i = 0; i < s.D; i += 2) {
                const double ang = (double)p / std::pow(10000.0, (double)i / (double)s.D);
                const double v2[2] = {std::sin(ang), std::cos(ang)};
                for (int k = 0; k < 2 && i + k < s.D; ++k) {
                    const size_t at = (size_t)p * s.D + i + k;
                    if (es == 2) {
                        const uint16_t b = tfm::bf16_bits_rne((float)v2[k]);
                        std::memcpy(host.data() + at * 2, &b, 2);
                    } else {
                        const float f = (float)v2[k];
                        std::memcpy(host.data() + at * 4, &f, 4);
                    }
                }
            }
        e = cudaMemcpy(m->pos, host.data(), host.size(), cudaMemcpyHostToDevice);
    }
    auto vec = [&](std::vector<float*>& dst, const void* const* src, int64_t n) {
        dst.assign(c.n_layer, nullptr);
        for (int l = 0; l < c.n_layer; ++l) {
            dst[l] = reinterpret_cast<float*>(take(n * 4));
            copy(dst[l], src[l], n * 4);
        }
    };
    auto mat = [&](std::vector<void*>& dst, const void* const* src, int64_t rows, int64_t cols) {
        dst.assign(c.n_layer, nullptr);
        for (int l = 0; l < c.n_layer; ++l) {
            dst[l] = take(rows * cols * es);
            copy(dst[l], src[l], rows * cols * es);
        }
    };
    if (c.n_layer > 0) {
        vec(m->attn_norm, w->ln1_g, s.D);
        vec(m->ln1_b, w->ln1_b, s.D);
        mat(m->wqkv, w->w_qkv, s.Nqkv, s.D);
        vec(m->b_qkv, w->b_qkv, s.Nqkv);
        mat(m->wo, w->w_proj, s.D, s.Dq);
        vec(m->b_proj, w->b_proj, s.D);
        vec(m->ffn_norm, w->ln2_g, s.D);
        vec(m->ln2_b, w->ln2_b, s.D);
        mat(m->w1, w->w_fc, s.F, s.D);
        vec(m->b_fc, w->b_fc, s.F);
        mat(m->w2, w->w_fc2, s.D, s.F);
        vec(m->b_fc2, w->b_fc2, s.D);
    }
    m->w3.assign(c.n_layer, nullptr);
    m->final_norm = reinterpret_cast<float*>(take(s.D * 4));
    copy(m->final_norm, w->lnf_g, s.D * 4);
    m->lnf_b = reinterpret_cast<float*>(take(s.D * 4));
    copy(m->lnf_b, w->lnf_b, s.D * 4);
    if (w->lm_head == w->embed) {
        m->lm_head = m->embed;
    } else {
        m->lm_head = take(s.V * s.D * es);
        copy(m->lm_head, w->lm_head, s.V * s.D * es);
    }
    m->lm_bias = nullptr;
    if (m->g2.lm_bias) {
        m->lm_bias = reinterpret_cast<float*>(take(s.V * 4));
        copy(m->lm_bias, w->lm_bias, s.V * 4);
    }
    if (over) return fail(TFM_EINVAL, "internal: weight storage overflow");
    if (e != cudaSuccess) return tfm::cuda_fail(e, "tfm_load_gpt2_weights");
    m->loaded = true;
    m->plan_m = -1;
    m->lse_M = -1;
    return TFM_OK;
}

}  // extern "C"

namespace tfm {
namespace {

EpiParams epi_basic(int kind, int M, int N, void* out, int64_t ldo) {
    EpiParams p{};
    p.kind = kind;
    p.M = M;
    p.N = N;
    p.out = out;
    p.ldo = ldo;
    return p;
}

EpiParams epi_qkv(Model* m, int M, int S) {
    const tfm_config& c = m->cfg;
    EpiParams p{};
    p.kind = EPI_QKV_ROPE;
    p.M = M;
    p.N = (int)m->sz.Nqkv;
    p.out_bf16 = c.mode == TFM_BF16;
    p.S = S;
    p.n_head = c.n_head;
    p.n_kv_head = c.n_kv_head;
    p.dh = c.d_model / c.n_head;
    p.rope_cs = m->rope();
    p.q = m->q();
    p.k = m->k();
    p.v = m->v();
    return p;
}

// (Re)builds the tensor maps of every tensor-core GEMM of the forward for M
// tokens of sequences of length S writing logits at (logits, ld).
tfm_status build_plans(Model* m, int M, int S, float* logits, int64_t ld) {
    if (m->plan_m == M && m->plan_S == S && m->plan_logits == logits && m->plan_ld == ld)
        return TFM_OK;
    const tfm_config& c = m->cfg;
    const auto& s = m->sz;
    m->p_qkv.resize(c.n_layer);
    m->p_o.resize(c.n_layer);
    m->p_gu.resize(c.n_layer);
    m->p_down.resize(c.n_layer);
    m->plan_m = -1;
    tfm_status st = TFM_OK;
    const bool g2 = m->arch == 1;   // GPT-2-style: biases, no RoPE, a GELU MLP
    for (int l = 0; l < c.n_layer && st == TFM_OK; ++l) {
        EpiParams eq = epi_qkv(m, M, S);
        if (g2) {
            eq.rope_cs = nullptr;
            eq.bias = m->b_qkv[l];
        }
        st = plan_gemm_tc(&m->p_qkv[l], m->xn(), s.D, m->wqkv[l], nullptr, s.D, M, (int)s.Nqkv,
                          (int)s.D, eq);
        EpiParams eo = epi_basic(EPI_ACCUM_F32, M, (int)s.D, m->h(), s.D);
        if (g2) eo.bias = m->b_proj[l];
        if (st == TFM_OK)
            st = plan_gemm_tc(&m->p_o[l], m->o(), s.Dq, m->wo[l], nullptr, s.Dq, M, (int)s.D,
                              (int)s.Dq, eo);
        if (st == TFM_OK) {
            EpiParams e = epi_basic(g2 ? EPI_GELU : EPI_SWIGLU, M, (int)s.F, m->a(), s.F);
            e.out_bf16 = 1;
            if (g2) e.bias = m->b_fc[l];
            st = plan_gemm_tc(&m->p_gu[l], m->xn(), s.D, m->w1[l], g2 ? nullptr : m->w3[l], s.D, M,
                              (int)s.F, (int)s.D, e);
        }
        EpiParams ed = epi_basic(EPI_ACCUM_F32, M, (int)s.D, m->h(), s.D);
        if (g2) ed.bias = m->b_fc2[l];
        if (st == TFM_OK)
            st = plan_gemm_tc(&m->p_down[l], m->a(), s.F, m->w2[l], nullptr, s.F, M, (int)s.D,
                              (int)s.F, ed);
    }
    EpiParams el = epi_basic(EPI_STORE_F32, M, (int)s.V, logits, ld);
    el.bias = m->lm_bias;
    if (st == TFM_OK)
        st = plan_gemm_tc(&m->p_lm, m->xn(), s.D, m->lm_head, nullptr, s.D, M, (int)s.V, (int)s.D, el);
    if (st != TFM_OK) return fail(st, "could not encode TMA tensor maps (driver entry point missing?)");
    // the model's weights: no launch writes them once loaded
    for (int l = 0; l < c.n_layer; ++l)
        m->p_qkv[l].b_static = m->p_o[l].b_static = m->p_gu[l].b_static = m->p_down[l].b_static = 1;
    m->p_lm.b_static = 1;
    m->plan_m = M;
    m->plan_S = S;
    const int dh = c.d_model / c.n_head;
    // (bf16 mode: every supported d_head, 32, 64 and 128, runs on tcgen05)
    if (plan_attention_tc(&m->p_attn, m->q(), m->k(), m->v(), m->o(), M / S, c.n_head,
                          c.n_kv_head, S, dh, 1.0f / std::sqrt((float)dh)) != TFM_OK) {
        m->plan_m = -1;
        return fail(TFM_ECUDA, "could not encode attention tensor maps");
    }
    m->plan_logits = logits;
    m->plan_ld = ld;
    return TFM_OK;
}

enum Kind { K_EMBED = 0, K_NORM, K_QKV, K_ATTN, K_OPROJ, K_GATEUP, K_DOWN, K_LMHEAD };

// Launch `expr`; when profiling, record an event after it and remember its kind.
#define TFM_LAUNCH(kind, expr)                                                  \
    do {                                                                        \
        cudaError_t _e = (expr);                                                \
        if (_e != cudaSuccess) return cuda_fail(_e, #expr);                     \
        if (run) {                                                              \
            cudaEvent_t _ev = m->next_event();                                  \
            if (!_ev) return fail(TFM_ECUDA, "cudaEventCreate failed");         \
            _e = cudaEventRecord(_ev, st);                                      \
            if (_e != cudaSuccess) return cuda_fail(_e, "cudaEventRecord");    \
            run->kinds.push_back(kind);                                         \
        }                                                                       \
    } while (0)

// Sliding window of layer l for sequences of length S: 0 when the layer attends
// to the whole prefix (no window, or a window of at least S positions).
int layer_window(const Model* m, int l, int S) {
    if (m->windows.empty()) return 0;
    const int w = m->windows[l];
    return (w > 0 && w < S) ? w : 0;
}

// Targets and outputs of tfm_forward_loss.
struct LossArgs {
    const int32_t* targets;
    float* loss;
    float* lse;
    float* mean;
};

int lse_slots_max(int V) { return 2 * ((V + 127) / 128); }

// Scratch of the fused cross-entropy for M rows (grown on demand).
tfm_status ensure_loss_scratch(Model* m, int64_t M) {
    if (m->loss_mem && m->loss_rows >= M) return TFM_OK;
    if (m->loss_mem) cudaFree(m->loss_mem);
    m->loss_mem = nullptr;
    m->loss_rows = 0;
    m->lse_M = -1;
    const int64_t V = m->cfg.vocab, ldV = (V + 3) / 4 * 4;
    const size_t part = (size_t)M * lse_slots_max((int)V) * 8, vec = (size_t)M * 4;
    const size_t lg = m->cfg.mode == TFM_BF16 ? 0 : (size_t)M * ldV * 4;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    cudaError_t e = cudaMalloc(&m->loss_mem, up(part) + 2 * up(vec) + lg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        m->loss_mem = nullptr;
        return fail(TFM_ENOMEM, "cross-entropy scratch for %lld rows: %s", (long long)M,
                    cudaGetErrorString(e));
    }
    m->lse_part = reinterpret_cast<float2*>(m->loss_mem);
    m->lse_tgt = reinterpret_cast<float*>(m->loss_mem + up(part));
    m->loss_tmp = reinterpret_cast<float*>(m->loss_mem + up(part) + up(vec));
    m->loss_logits = lg ? reinterpret_cast<float*>(m->loss_mem + up(part) + 2 * up(vec)) : nullptr;
    m->loss_rows = M;
    return TFM_OK;
}

// The LM head as the fused cross-entropy's GEMM: statistics instead of logits.
tfm_status build_lse_plan(Model* m, int M, const int32_t* targets) {
    if (m->lse_M == M && m->lse_targets == targets) return TFM_OK;
    const auto& s = m->sz;
    EpiParams e = epi_basic(EPI_LSE, M, (int)s.V, nullptr, 0);
    e.bias = m->lm_bias;
    e.targets = targets;
    e.lse_part = m->lse_part;
    e.lse_tgt = m->lse_tgt;
    m->lse_M = -1;
    tfm_status st = plan_gemm_tc(&m->p_lse, m->xn(), s.D, m->lm_head, nullptr, s.D, M, (int)s.V,
                                 (int)s.D, e);
    if (st != TFM_OK) return fail(st, "could not encode TMA tensor maps (driver entry point missing?)");
    // slot 2 * column tile + half; at most lse_slots_max(V) for tiles of >= 128 columns
    m->p_lse.epi.lse_slots = 2 * (int)((s.V + m->p_lse.block_n - 1) / m->p_lse.block_n);
    m->p_lse.b_static = 1;
    m->lse_M = M;
    m->lse_targets = targets;
    return TFM_OK;
}

tfm_status forward_impl(Model* m, const int32_t* tokens, int B, int S, float* logits, int64_t ld,
                        cudaStream_t st, bool to_cache = false, const LossArgs* la = nullptr) {
    const tfm_config& c = m->cfg;
    const auto& s = m->sz;
    const int M = B * S;
    const int dh = c.d_model / c.n_head;
    const float scale = 1.0f / std::sqrt((float)dh);
    const bool bf = c.mode == TFM_BF16;
    if (!device_error_word()) return fail(TFM_ECUDA, "device error word unavailable");
    if (la) {
        tfm_status ls = ensure_loss_scratch(m, M);
        if (ls != TFM_OK) return ls;
        if (bf) {
            ls = build_lse_plan(m, M, la->targets);
            if (ls != TFM_OK) return ls;
        }
        // the logits plan is not launched: keep the one already built for (M, S)
        if (m->plan_m == M && m->plan_S == S) {
            logits = const_cast<float*>(m->plan_logits);
            ld = m->plan_ld;
        } else {
            logits = nullptr;
            ld = 0;
        }
    }
    if (bf) {
        tfm_status ps = build_plans(m, M, S, logits, ld);
        if (ps != TFM_OK) return ps;
    }
    Model::ProfRun* run = nullptr;
    if (m->prof) {
        m->runs.push_back(Model::ProfRun{m->ev_used, {}});
        run = &m->runs.back();
        cudaEvent_t ev = m->next_event();
        if (!ev) return fail(TFM_ECUDA, "cudaEventCreate failed");
        cudaError_t re = cudaEventRecord(ev, st);
        if (re != cudaSuccess) return cuda_fail(re, "cudaEventRecord");
    }
    // The GPT-2-style family: LayerNorm (gain, shift), position rows in the
    // embedding, post-norm blocks normalising the residual stream in place.
    const bool g2 = m->arch == 1;
    const bool post = g2 && m->g2.post_norm;
    auto ln_args = [&](const float* b, float* h_out) {
        NormArgs n{};
        n.kind = kNormLayer;
        n.b = b;
        n.h_out = h_out;
        return n;
    };
    // Embedding and the first norm (layer 0's input norm, or the final norm of a
    // model without layers; none before a post-norm block) in one pass.
    NormArgs na0{};
    if (g2) {
        if (c.n_layer == 0) na0 = ln_args(m->lnf_b, nullptr);
        else if (post) na0.kind = kNormNone;
        else na0 = ln_args(m->ln1_b[0], nullptr);
        na0.pos = m->pos;
        na0.S = S;
    }
    TFM_LAUNCH(K_EMBED, launch_embed_rmsnorm(tokens, m->embed,
                                             c.n_layer > 0 ? m->attn_norm[0] : m->final_norm,
                                             m->h(), m->xn(), M, c.vocab, c.d_model, c.norm_eps,
                                             bf, st, 1, g2 ? &na0 : nullptr));
    // the norms of a layer: before the attention (pre-norm, l > 0), after the
    // output projection (post-norm LN1 in place, or the pre-norm FFN input), after
    // the MLP (post-norm LN2 in place)
    auto norm_pre_attn = [&](int l) -> cudaError_t {
        NormArgs n = g2 ? ln_args(m->ln1_b[l], nullptr) : NormArgs{};
        return launch_rmsnorm(m->h(), m->attn_norm[l], m->xn(), M, c.d_model, c.norm_eps, bf, st, 1,
                              g2 ? &n : nullptr);
    };
    auto norm_mid = [&](int l) -> cudaError_t {
        NormArgs n = post ? ln_args(m->ln1_b[l], m->h())
                          : (g2 ? ln_args(m->ln2_b[l], nullptr) : NormArgs{});
        return launch_rmsnorm(m->h(), post ? m->attn_norm[l] : m->ffn_norm[l], m->xn(), M,
                              c.d_model, c.norm_eps, bf, st, 1, g2 ? &n : nullptr);
    };
    auto norm_post_mlp = [&](int l) -> cudaError_t {
        NormArgs n = ln_args(m->ln2_b[l], m->h());
        return launch_rmsnorm(m->h(), m->ffn_norm[l], m->xn(), M, c.d_model, c.norm_eps, bf, st, 1, &n);
    };
    auto norm_final = [&]() -> cudaError_t {
        NormArgs n = g2 ? ln_args(m->lnf_b, nullptr) : NormArgs{};
        return launch_rmsnorm(m->h(), m->final_norm, m->xn(), M, c.d_model, c.norm_eps, bf, st, 1,
                              g2 ? &n : nullptr);
    };
    if (bf) {
        for (int l = 0; l < c.n_layer; ++l) {
            if (l > 0 && !post) TFM_LAUNCH(K_NORM, norm_pre_attn(l));
            TFM_LAUNCH(K_QKV, launch_gemm_tc(m->p_qkv[l], st));
            if (to_cache) {
                // k, v of positions [0, S) into the layer's cache: rows (b, kv head)
                // of S*dh elements, cache row pitch max_seq*dh.
                const size_t row = (size_t)S * dh * 2, pitch = (size_t)c.max_seq * dh * 2;
                const size_t rows = (size_t)B * c.n_kv_head;
                cudaError_t e = cudaMemcpy2DAsync(m->kcache(l), pitch, m->k(), row, row, rows,
                                                  cudaMemcpyDeviceToDevice, st);
                if (e == cudaSuccess)
                    e = cudaMemcpy2DAsync(m->vcache(l), pitch, m->v(), row, row, rows,
                                          cudaMemcpyDeviceToDevice, st);
                if (e != cudaSuccess) return cuda_fail(e, "k, v into the cache");
            }
            // a sliding-window layer (window < S) skips the key tiles before each
            // query tile's window and masks the band's edge
            const int win = layer_window(m, l, S);
            {
                AttnPlan pw = m->p_attn;
                pw.window = win;
                TFM_LAUNCH(K_ATTN, launch_attention_tc(pw, st));
            }
            TFM_LAUNCH(K_OPROJ, launch_gemm_tc(m->p_o[l], st));
            TFM_LAUNCH(K_NORM, norm_mid(l));
            TFM_LAUNCH(K_GATEUP, launch_gemm_tc(m->p_gu[l], st));
            TFM_LAUNCH(K_DOWN, launch_gemm_tc(m->p_down[l], st));
            if (post) TFM_LAUNCH(K_NORM, norm_post_mlp(l));
        }
        if (c.n_layer > 0) TFM_LAUNCH(K_NORM, norm_final());
        if (la) {
            TFM_LAUNCH(K_LMHEAD, launch_gemm_tc(m->p_lse, st));
            TFM_LAUNCH(K_LMHEAD, launch_lse_finish(m->lse_part, m->p_lse.epi.lse_slots, m->lse_tgt,
                                                   la->targets, M, c.vocab, la->loss, la->lse,
                                                   m->loss_tmp, la->mean, st));
        } else {
            TFM_LAUNCH(K_LMHEAD, launch_gemm_tc(m->p_lm, st));
        }
    } else {
        const float* xn = static_cast<const float*>(m->xn());
        for (int l = 0; l < c.n_layer; ++l) {
            if (l > 0 && !post) TFM_LAUNCH(K_NORM, norm_pre_attn(l));
            EpiParams eq = epi_qkv(m, M, S);
            if (g2) {
                eq.rope_cs = nullptr;
                eq.bias = m->b_qkv[l];
            }
            TFM_LAUNCH(K_QKV, launch_gemm_simt(xn, static_cast<const float*>(m->wqkv[l]), nullptr, M,
                                               (int)s.Nqkv, c.d_model, eq, st));
            TFM_LAUNCH(K_ATTN, launch_attention_simt(static_cast<const float*>(m->q()),
                                                     static_cast<const float*>(m->k()),
                                                     static_cast<const float*>(m->v()),
                                                     static_cast<float*>(m->o()), B, c.n_head,
                                                     c.n_kv_head, S, dh, scale, st,
                                                     layer_window(m, l, S)));
            EpiParams eo = epi_basic(EPI_ACCUM_F32, M, c.d_model, m->h(), s.D);
            if (g2) eo.bias = m->b_proj[l];
            TFM_LAUNCH(K_OPROJ, launch_gemm_simt(static_cast<const float*>(m->o()),
                                                 static_cast<const float*>(m->wo[l]), nullptr, M,
                                                 c.d_model, (int)s.Dq, eo, st));
            TFM_LAUNCH(K_NORM, norm_mid(l));
            EpiParams e = epi_basic(g2 ? EPI_GELU : EPI_SWIGLU, M, c.d_ff, m->a(), s.F);
            e.out_bf16 = 0;
            if (g2) e.bias = m->b_fc[l];
            TFM_LAUNCH(K_GATEUP, launch_gemm_simt(xn, static_cast<const float*>(m->w1[l]),
                                                  g2 ? nullptr : static_cast<const float*>(m->w3[l]),
                                                  M, c.d_ff, c.d_model, e, st));
            EpiParams ed = epi_basic(EPI_ACCUM_F32, M, c.d_model, m->h(), s.D);
            if (g2) ed.bias = m->b_fc2[l];
            TFM_LAUNCH(K_DOWN, launch_gemm_simt(static_cast<const float*>(m->a()),
                                                static_cast<const float*>(m->w2[l]), nullptr, M,
                                                c.d_model, c.d_ff, ed, st));
            if (post) TFM_LAUNCH(K_NORM, norm_post_mlp(l));
        }
        if (c.n_layer > 0) TFM_LAUNCH(K_NORM, norm_final());
        EpiParams el = epi_basic(EPI_STORE_F32, M, c.vocab, logits, ld);
        el.bias = m->lm_bias;
        if (la) {
            // fp32 mode: the logits in scratch, then one pass over each row
            const int64_t ldV = (c.vocab + 3) / 4 * 4;
            el.out = m->loss_logits;
            el.ldo = ldV;
            TFM_LAUNCH(K_LMHEAD, launch_gemm_simt(xn, static_cast<const float*>(m->lm_head), nullptr, M,
                                                  c.vocab, c.d_model, el, st));
            TFM_LAUNCH(K_LMHEAD, launch_lse_rows(m->loss_logits, ldV, M, c.vocab, la->targets,
                                                 m->lse_part, m->lse_tgt, st));
            TFM_LAUNCH(K_LMHEAD, launch_lse_finish(m->lse_part, 1, m->lse_tgt, la->targets, M,
                                                   c.vocab, la->loss, la->lse, m->loss_tmp, la->mean,
                                                   st));
        } else {
            TFM_LAUNCH(K_LMHEAD, launch_gemm_simt(xn, static_cast<const float*>(m->lm_head), nullptr, M,
                                                  c.vocab, c.d_model, el, st));
        }
    }
    return TFM_OK;
}

// Tensor-core plans of a decode step: M = B rows (one new token per sequence),
// q, k, v of that token head-major with S = 1; the RoPE position is set per step.
tfm_status build_decode_plans(Model* m, int B, float* logits, int64_t ld) {
    if (m->dplan_B == B && m->dplan_logits == logits && m->dplan_ld == ld) return TFM_OK;
    const tfm_config& c = m->cfg;
    const auto& s = m->sz;
    m->d_qkv.resize(c.n_layer);
    m->d_o.resize(c.n_layer);
    m->d_gu.resize(c.n_layer);
    m->d_down.resize(c.n_layer);
    m->dplan_B = -1;
    tfm_status st = TFM_OK;
    const bool g2 = m->arch == 1;   // GPT-2-style: biases, no RoPE, a GELU MLP
    for (int l = 0; l < c.n_layer && st == TFM_OK; ++l) {
        {
            // k and v of the new token go straight into the layer's cache
            EpiParams e = epi_qkv(m, B, 1);
            e.k = m->kcache(l);
            e.v = m->vcache(l);
            e.kv_stride = c.max_seq;
            e.pos0_dev = m->pos_dev;        // RoPE and cache position of the step
            if (g2) {
                e.rope_cs = nullptr;
                e.bias = m->b_qkv[l];
            }
            st = plan_gemm_tc(&m->d_qkv[l], m->xn(), s.D, m->wqkv[l], nullptr, s.D, B,
                              (int)s.Nqkv, (int)s.D, e);
        }
        EpiParams eo = epi_basic(EPI_ACCUM_F32, B, (int)s.D, m->h(), s.D);
        if (g2) eo.bias = m->b_proj[l];
        if (st == TFM_OK)
            st = plan_gemm_tc(&m->d_o[l], m->o(), s.Dq, m->wo[l], nullptr, s.Dq, B, (int)s.D,
                              (int)s.Dq, eo);
        if (st == TFM_OK) {
            EpiParams e = epi_basic(g2 ? EPI_GELU : EPI_SWIGLU, B, (int)s.F, m->a(), s.F);
            e.out_bf16 = 1;
            if (g2) e.bias = m->b_fc[l];
            st = plan_gemm_tc(&m->d_gu[l], m->xn(), s.D, m->w1[l], g2 ? nullptr : m->w3[l], s.D, B,
                              (int)s.F, (int)s.D, e);
        }
        EpiParams ed = epi_basic(EPI_ACCUM_F32, B, (int)s.D, m->h(), s.D);
        if (g2) ed.bias = m->b_fc2[l];
        if (st == TFM_OK)
            st = plan_gemm_tc(&m->d_down[l], m->a(), s.F, m->w2[l], nullptr, s.F, B, (int)s.D,
                              (int)s.F, ed);
    }
    EpiParams el = epi_basic(EPI_STORE_F32, B, (int)s.V, logits, ld);
    el.bias = m->lm_bias;
    if (st == TFM_OK)
        st = plan_gemm_tc(&m->d_lm, m->xn(), s.D, m->lm_head, nullptr, s.D, B, (int)s.V, (int)s.D, el);
    if (st != TFM_OK) return fail(st, "could not encode TMA tensor maps (driver entry point missing?)");
    for (int l = 0; l < c.n_layer; ++l)
        m->d_qkv[l].b_static = m->d_o[l].b_static = m->d_gu[l].b_static = m->d_down[l].b_static = 1;
    m->d_lm.b_static = 1;
    // RMSNorm models with up to 16 sequences: the weight-streaming GEMMs after
    // each norm take the residual rows and normalise them on the way in, so the
    // step has no norm launches after the first (fused with the embedding).
    m->dnorm_fused = !g2 && c.n_layer > 0 && m->d_lm.skinny && m->d_lm.sk_nm == 16;
    for (int l = 0; l < c.n_layer && m->dnorm_fused; ++l)
        m->dnorm_fused = m->d_qkv[l].skinny && m->d_qkv[l].sk_nm == 16 && m->d_gu[l].skinny &&
                         m->d_gu[l].sk_nm == 16;
    if (m->dnorm_fused) {
        for (int l = 0; l < c.n_layer; ++l) {
            if (l > 0) {
                m->d_qkv[l].norm_x = m->h();
                m->d_qkv[l].norm_g = m->attn_norm[l];
                m->d_qkv[l].norm_eps = c.norm_eps;
            }
            m->d_gu[l].norm_x = m->h();
            m->d_gu[l].norm_g = m->ffn_norm[l];
            m->d_gu[l].norm_eps = c.norm_eps;
        }
        m->d_lm.norm_x = m->h();
        m->d_lm.norm_g = m->final_norm;
        m->d_lm.norm_eps = c.norm_eps;
    }
    m->dplan_B = B;
    m->dplan_logits = logits;
    m->dplan_ld = ld;
    return TFM_OK;
}

// One decode step: token t_b of every sequence b at position *pos_dev, the cache
// holding positions [0, *pos_dev).  The same blocks as the forward with M = B;
// each layer writes the token's k, v into its cache (from the QKV epilogue) and
// attends over [0, *pos_dev].  Nothing here depends on the position on the host,
// so the launches can be recorded once and replayed at every position.
tfm_status decode_body(Model* m, const int32_t* tokens, int B, float* logits, int64_t ld,
                       cudaStream_t st) {
    const tfm_config& c = m->cfg;
    const int dh = c.d_model / c.n_head;
    const float scale = 1.0f / std::sqrt((float)dh);
    if (!device_error_word()) return fail(TFM_ECUDA, "device error word unavailable");
    tfm_status ps = build_decode_plans(m, B, logits, ld);
    if (ps != TFM_OK) return ps;
    Model::ProfRun* run = nullptr;
    if (m->prof) {
        m->runs.push_back(Model::ProfRun{m->ev_used, {}});
        run = &m->runs.back();
        cudaEvent_t ev = m->next_event();
        if (!ev) return fail(TFM_ECUDA, "cudaEventCreate failed");
        cudaError_t re = cudaEventRecord(ev, st);
        if (re != cudaSuccess) return cuda_fail(re, "cudaEventRecord");
    }
    // The GPT-2-style family: LayerNorm, the position row of the step added in
    // the embedding, post-norm blocks normalising the residual stream in place.
    const bool g2 = m->arch == 1;
    const bool post = g2 && m->g2.post_norm;
    auto ln_args = [&](const float* bb, float* h_out) {
        NormArgs n{};
        n.kind = kNormLayer;
        n.b = bb;
        n.h_out = h_out;
        return n;
    };
    NormArgs na0{};
    if (g2) {
        if (c.n_layer == 0) na0 = ln_args(m->lnf_b, nullptr);
        else if (post) na0.kind = kNormNone;
        else na0 = ln_args(m->ln1_b[0], nullptr);
        na0.pos = m->pos;
        na0.S = 1;
        na0.pos_dev = m->pos_dev;
    }
    TFM_LAUNCH(K_EMBED, launch_embed_rmsnorm(tokens, m->embed,
                                             c.n_layer > 0 ? m->attn_norm[0] : m->final_norm,
                                             m->h(), m->xn(), B, c.vocab, c.d_model, c.norm_eps,
                                             1, st, 1, g2 ? &na0 : nullptr));
    auto norm = [&](const float* gain, const NormArgs* n) {
        return launch_rmsnorm(m->h(), gain, m->xn(), B, c.d_model, c.norm_eps, 1, st, 1, n);
    };
    for (int l = 0; l < c.n_layer; ++l) {
        if (l > 0 && !post && !m->dnorm_fused) {
            NormArgs n = ln_args(g2 ? m->ln1_b[l] : nullptr, nullptr);
            TFM_LAUNCH(K_NORM, norm(m->attn_norm[l], g2 ? &n : nullptr));
        }
        TFM_LAUNCH(K_QKV, launch_gemm_tc(m->d_qkv[l], st));
        TFM_LAUNCH(K_ATTN, launch_decode_attention(m->q(), m->kcache(l), m->vcache(l), m->dec_part,
                                                   m->o(), B, c.n_head, c.n_kv_head, c.max_seq,
                                                   m->pos_dev, dh, scale, st,
                                                   m->windows.empty() ? 0 : m->windows[l]));
        TFM_LAUNCH(K_OPROJ, launch_gemm_tc(m->d_o[l], st));
        if (!m->dnorm_fused) {
            NormArgs n = post ? ln_args(m->ln1_b[l], m->h())
                              : ln_args(g2 ? m->ln2_b[l] : nullptr, nullptr);
            TFM_LAUNCH(K_NORM, norm(post ? m->attn_norm[l] : m->ffn_norm[l], g2 ? &n : nullptr));
        }
        TFM_LAUNCH(K_GATEUP, launch_gemm_tc(m->d_gu[l], st));
        TFM_LAUNCH(K_DOWN, launch_gemm_tc(m->d_down[l], st));
        if (post) {
            NormArgs n = ln_args(m->ln2_b[l], m->h());
            TFM_LAUNCH(K_NORM, norm(m->ffn_norm[l], &n));
        }
    }
    if (c.n_layer > 0 && !m->dnorm_fused) {
        NormArgs n = ln_args(g2 ? m->lnf_b : nullptr, nullptr);
        TFM_LAUNCH(K_NORM, norm(m->final_norm, g2 ? &n : nullptr));
    }
    TFM_LAUNCH(K_LMHEAD, launch_gemm_tc(m->d_lm, st));
    return TFM_OK;
}

// The step at position pos: the position and the tokens are stored on the
// device, then the body runs.  A step with the same batch, logits and stream as
// the previous one is recorded once and replayed from then on (not when
// profiling, nor on the legacy stream, which cannot be captured).
tfm_status decode_impl(Model* m, const int32_t* tokens, int B, int pos, float* logits, int64_t ld,
                       cudaStream_t st) {
    cudaError_t e = launch_decode_setup(m->pos_dev, pos, tokens, m->tok_dev, B, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode setup");
    if (m->prof || !st) return decode_body(m, m->tok_dev, B, logits, ld, st);
    Model::Graph* g = nullptr;
    for (auto& c : m->dgraphs)
        if (c.exec && c.B == B && c.logits == logits && c.ld == ld && c.stream == (void*)st) g = &c;
    if (!g) {
        Model::Graph& last = m->dlast;
        const bool again = last.B == B && last.logits == logits && last.ld == ld && last.stream == (void*)st;
        last.B = B;
        last.logits = logits;
        last.ld = ld;
        last.stream = st;
        if (!again) return decode_body(m, m->tok_dev, B, logits, ld, st);
        g = &m->dgraphs[0];
        for (auto& c : m->dgraphs)
            if (!c.exec || c.used < g->used) g = &c;
        if (g->exec) {
            cudaGraphExecDestroy(g->exec);
            g->exec = nullptr;
        }
        e = cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal);
        if (e != cudaSuccess) return cuda_fail(e, "begin capture");
        tfm_status ts = decode_body(m, m->tok_dev, B, logits, ld, st);
        cudaGraph_t graph = nullptr;
        e = cudaStreamEndCapture(st, &graph);
        if (ts != TFM_OK || e != cudaSuccess) {
            if (graph) cudaGraphDestroy(graph);
            return ts != TFM_OK ? ts : cuda_fail(e, "end capture");
        }
        e = cudaGraphInstantiate(&g->exec, graph, 0);
        cudaGraphDestroy(graph);
        if (e != cudaSuccess) {
            g->exec = nullptr;
            return cuda_fail(e, "graph instantiate");
        }
        g->B = B;
        g->logits = logits;
        g->ld = ld;
        g->stream = st;
    }
    g->used = ++m->graph_clock;
    e = cudaGraphLaunch(g->exec, st);
    return e == cudaSuccess ? TFM_OK : cuda_fail(e, "graph launch");
}

tfm_status check_forward_args(Model* m, const void* tokens, int B, int S, const float* logits,
                              int64_t ld) {
    if (!m) return fail(TFM_EINVAL, "NULL handle");
    if (!m->loaded) return fail(TFM_EINVAL, "weights not loaded");
    if (!tokens || !logits) return fail(TFM_EINVAL, "NULL tokens or logits");
    if (!aligned_to(tokens, 4)) return fail(TFM_EINVAL, "tokens must be 4-byte aligned");
    if (B < 1 || B > m->cfg.max_batch) return fail(TFM_EINVAL, "B=%d outside [1, max_batch=%d]", B, m->cfg.max_batch);
    if (S < 1 || S > m->cfg.max_seq) return fail(TFM_EINVAL, "S=%d outside [1, max_seq=%d]", S, m->cfg.max_seq);
    if (ld < m->cfg.vocab || ld % 4) return fail(TFM_EINVAL, "ld_logits=%lld must be >= vocab and a multiple of 4", (long long)ld);
    return TFM_OK;
}

}  // namespace
}  // namespace tfm

extern "C" {

tfm_status tfm_forward(void* handle, const int32_t* tokens, int32_t B, int32_t S, float* logits,
                       int64_t ld_logits, void* stream) {
    Model* m = static_cast<Model*>(handle);
    tfm_status st = tfm::check_forward_args(m, tokens, B, S, logits, ld_logits);
    if (st != TFM_OK) return st;
    if (!tfm::aligned16(logits)) return fail(TFM_EINVAL, "logits must be 16-byte aligned");
    return tfm::forward_impl(m, tokens, B, S, logits, ld_logits, static_cast<cudaStream_t>(stream));
}

tfm_status tfm_forward_loss(void* handle, const int32_t* tokens, const int32_t* targets, int32_t B,
                            int32_t S, float* loss, float* lse, float* mean_loss, void* stream) {
    Model* m = static_cast<Model*>(handle);
    if (!m) return fail(TFM_EINVAL, "NULL handle");
    if (!targets) return fail(TFM_EINVAL, "NULL targets");
    if (!tfm::aligned_to(targets, 4) || !tfm::aligned_to(loss, 4) || !tfm::aligned_to(lse, 4) ||
        !tfm::aligned_to(mean_loss, 4))
        return fail(TFM_EINVAL, "targets, loss, lse and mean_loss must be 4-byte aligned");
    // the logits-free forward takes the same token checks as tfm_forward
    const float dummy = 0.f;
    tfm_status st = tfm::check_forward_args(m, tokens, B, S, &dummy, (m->cfg.vocab + 3) / 4 * 4);
    if (st != TFM_OK) return st;
    const tfm::LossArgs la{targets, loss, lse, mean_loss};
    return tfm::forward_impl(m, tokens, B, S, nullptr, 0, static_cast<cudaStream_t>(stream), false,
                             &la);
}

tfm_status tfm_set_attention_windows(void* handle, const int32_t* windows, int32_t n) {
    Model* m = static_cast<Model*>(handle);
    if (!m) return fail(TFM_EINVAL, "NULL handle");
    if (n != 0 && n != m->cfg.n_layer) return fail(TFM_EINVAL, "n must be 0 or n_layer (%d)", m->cfg.n_layer);
    if (n > 0 && !windows) return fail(TFM_EINVAL, "NULL windows");
    for (int l = 0; l < n; ++l)
        if (windows[l] < 0) return fail(TFM_EINVAL, "window of layer %d is negative", l);
    // recorded forwards and decode steps hold the previous windows
    for (auto& g : m->graphs)
        if (g.exec) {
            cudaGraphExecDestroy(g.exec);
            g = Model::Graph{};
        }
    for (auto& g : m->dgraphs)
        if (g.exec) {
            cudaGraphExecDestroy(g.exec);
            g = Model::Graph{};
        }
    m->dlast = Model::Graph{};
    m->windows.assign(windows, windows + n);
    return TFM_OK;
}

}  // extern "C"

namespace tfm {
namespace {

// Device -> host copy of the logits of M rows from an internal buffer (row
// stride ldV): one contiguous copy when the host rows have the same stride (the
// padding columns [vocab, ldV) are zeros), else a pitched copy of the vocab
// columns only (a row of vocab fp32 values need not be a multiple of 16 bytes,
// which slows the pitched copy).
cudaError_t copy_logits_to_host(Model* m, float* host, int64_t ld, const float* dev, int64_t M,
                                cudaStream_t st) {
    if (ld == m->sz.ldV)
        return cudaMemcpyAsync(host, dev, (size_t)M * ld * 4, cudaMemcpyDeviceToHost, st);
    return cudaMemcpy2DAsync(host, ld * 4, dev, m->sz.ldV * 4, (size_t)m->cfg.vocab * 4, M,
                             cudaMemcpyDeviceToHost, st);
}

// Launches the forward for these arguments from a recorded graph, recording it
// first if no kept recording matches (the least recently used one is replaced).
tfm_status graph_forward(Model* m, const int32_t* tokens, int B, int S, float* logits, int64_t ld,
                         cudaStream_t cs) {
    Model::Graph* g = nullptr;
    for (auto& c : m->graphs)
        if (c.exec && c.tokens == tokens && c.B == B && c.S == S && c.logits == logits &&
            c.ld == ld && c.stream == (void*)cs)
            g = &c;
    if (!g) {
        g = &m->graphs[0];
        for (auto& c : m->graphs)
            if (!c.exec || c.used < g->used) g = &c;
        if (g->exec) {
            cudaGraphExecDestroy(g->exec);
            g->exec = nullptr;
        }
        const bool prof = m->prof;
        m->prof = false;
        cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
        if (e != cudaSuccess) {
            m->prof = prof;
            return cuda_fail(e, "begin capture");
        }
        tfm_status st = forward_impl(m, tokens, B, S, logits, ld, cs);
        cudaGraph_t graph = nullptr;
        e = cudaStreamEndCapture(cs, &graph);
        m->prof = prof;
        if (st != TFM_OK || e != cudaSuccess) {
            if (graph) cudaGraphDestroy(graph);
            return st != TFM_OK ? st : cuda_fail(e, "end capture");
        }
        e = cudaGraphInstantiate(&g->exec, graph, 0);
        cudaGraphDestroy(graph);
        if (e != cudaSuccess) {
            g->exec = nullptr;
            return cuda_fail(e, "graph instantiate");
        }
        g->tokens = tokens;
        g->B = B;
        g->S = S;
        g->logits = logits;
        g->ld = ld;
        g->stream = cs;
    }
    g->used = ++m->graph_clock;
    const cudaError_t e = cudaGraphLaunch(g->exec, cs);
    return e == cudaSuccess ? TFM_OK : cuda_fail(e, "graph launch");
}

}  // namespace
}  // namespace tfm

extern "C" {

tfm_status tfm_forward_graph(void* handle, const int32_t* tokens, int32_t B, int32_t S,
                             float* logits, int64_t ld_logits, void* stream) {
    Model* m = static_cast<Model*>(handle);
    tfm_status st = tfm::check_forward_args(m, tokens, B, S, logits, ld_logits);
    if (st != TFM_OK) return st;
    if (!tfm::aligned16(logits)) return fail(TFM_EINVAL, "logits must be 16-byte aligned");
    if (!stream) return fail(TFM_EINVAL, "tfm_forward_graph needs a non-default stream");
    return tfm::graph_forward(m, tokens, B, S, logits, ld_logits, static_cast<cudaStream_t>(stream));
}

tfm_status tfm_forward_host_async(void* handle, const int32_t* tokens_host, int32_t B, int32_t S,
                                  float* logits_host, int64_t ld_logits, void* stream) {
    Model* m = static_cast<Model*>(handle);
    tfm_status st = tfm::check_forward_args(m, tokens_host, B, S, logits_host, ld_logits);
    if (st != TFM_OK) return st;
    if (!stream) return fail(TFM_EINVAL, "tfm_forward_host_async needs a non-default stream");
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const int b = (int)(m->async_calls & 1);
    const int64_t M = (int64_t)B * S;
    // Buffer b is written again only once the copy that last read it is done.
    cudaError_t e = m->copy_pending[b] ? cudaStreamWaitEvent(cs, m->copied[b], 0) : cudaSuccess;
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(m->tok(), tokens_host, M * 4, cudaMemcpyHostToDevice, cs);
    if (e != cudaSuccess) return tfm::cuda_fail(e, "tokens host->device");
    st = tfm::graph_forward(m, m->tok(), B, S, m->logits_buf(b), m->sz.ldV, cs);
    if (st != TFM_OK) return st;
    e = cudaEventRecord(m->fwd_done[b], cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(m->copy_st, m->fwd_done[b], 0);
    if (e == cudaSuccess)
        e = tfm::copy_logits_to_host(m, logits_host, ld_logits, m->logits_buf(b), M, m->copy_st);
    if (e == cudaSuccess) e = cudaEventRecord(m->copied[b], m->copy_st);
    if (e != cudaSuccess) return tfm::cuda_fail(e, "logits device->host");
    m->copy_pending[b] = true;
    ++m->async_calls;
    return TFM_OK;
}

tfm_status tfm_kv_cache_create(void* handle) {
    Model* m = static_cast<Model*>(handle);
    if (!m) return fail(TFM_EINVAL, "NULL handle");
    if (m->kv) return TFM_OK;
    const tfm_config& c = m->cfg;
    const int dh = c.d_model / c.n_head;
    if (c.mode != TFM_BF16) return fail(TFM_EUNSUPPORTED, "the KV cache needs bf16 mode");
    if (!tfm::decode_supported(dh, c.n_head / c.n_kv_head))
        return fail(TFM_EUNSUPPORTED, "decode needs d_head in {32, 64, 128} and H/Hkv in {1, 2, 4, 8, 16} (<= 8 at d_head 128)");
    const size_t layer = (size_t)c.max_batch * c.n_kv_head * c.max_seq * dh * 2;
    const size_t caches = (size_t)c.n_layer * 2 * layer;
    const size_t part = tfm::decode_partial_floats(c.max_batch, c.n_head, c.max_seq, dh) * 4;
    uint8_t* p = nullptr;
    const cudaError_t e = cudaMalloc(&p, caches + part + 512 + (size_t)c.max_batch * 4);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(TFM_ENOMEM, "KV cache of %zu bytes: %s", caches + part, cudaGetErrorString(e));
    }
    m->kv = p;
    m->kv_layer_bytes = layer;
    m->dec_part = reinterpret_cast<float*>(p + (caches + 255) / 256 * 256);
    m->pos_dev = reinterpret_cast<int*>(p + (caches + 255) / 256 * 256 + (part + 255) / 256 * 256);
    m->tok_dev = m->pos_dev + 4;
    m->kv_len = 0;
    m->kv_batch = 0;
    return TFM_OK;
}

tfm_status tfm_prefill(void* handle, const int32_t* tokens, int32_t B, int32_t S, float* logits,
                       int64_t ld_logits, void* stream) {
    Model* m = static_cast<Model*>(handle);
    tfm_status st = tfm::check_forward_args(m, tokens, B, S, logits, ld_logits);
    if (st != TFM_OK) return st;
    if (!tfm::aligned16(logits)) return fail(TFM_EINVAL, "logits must be 16-byte aligned");
    if (!m->kv) return fail(TFM_EINVAL, "no KV cache: call tfm_kv_cache_create first");
    st = tfm::forward_impl(m, tokens, B, S, logits, ld_logits, static_cast<cudaStream_t>(stream),
                           true);
    if (st != TFM_OK) return st;
    m->kv_len = S;
    m->kv_batch = B;
    return TFM_OK;
}

tfm_status tfm_decode_step(void* handle, const int32_t* tokens, int32_t B, int32_t pos,
                           float* logits, int64_t ld_logits, void* stream) {
    Model* m = static_cast<Model*>(handle);
    tfm_status st = tfm::check_forward_args(m, tokens, B, 1, logits, ld_logits);
    if (st != TFM_OK) return st;
    if (!tfm::aligned16(logits)) return fail(TFM_EINVAL, "logits must be 16-byte aligned");
    if (!m->kv) return fail(TFM_EINVAL, "no KV cache: call tfm_kv_cache_create first");
    if (m->kv_batch != B) return fail(TFM_EINVAL, "B=%d differs from the cached batch %d", B, m->kv_batch);
    if (pos != m->kv_len) return fail(TFM_EINVAL, "pos=%d must equal the cached length %d", pos, m->kv_len);
    if (pos >= m->cfg.max_seq) return fail(TFM_EINVAL, "pos=%d reaches max_seq=%d", pos, m->cfg.max_seq);
    st = tfm::decode_impl(m, tokens, B, pos, logits, ld_logits, static_cast<cudaStream_t>(stream));
    if (st != TFM_OK) return st;
    m->kv_len = pos + 1;
    return TFM_OK;
}

tfm_status tfm_forward_host_join(void* handle, void* stream) {
    Model* m = static_cast<Model*>(handle);
    if (!m) return fail(TFM_EINVAL, "NULL handle");
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    for (int b = 0; b < 2; ++b)
        if (m->copy_pending[b]) {
            const cudaError_t e = cudaStreamWaitEvent(cs, m->copied[b], 0);
            if (e != cudaSuccess) return tfm::cuda_fail(e, "join copies");
        }
    return TFM_OK;
}

tfm_status tfm_forward_host(void* handle, const int32_t* tokens_host, int32_t B, int32_t S,
                            float* logits_host, int64_t ld_logits, void* stream) {
    Model* m = static_cast<Model*>(handle);
    tfm_status st = tfm::check_forward_args(m, tokens_host, B, S, logits_host, ld_logits);
    if (st != TFM_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const int64_t M = (int64_t)B * S;
    cudaError_t e = cudaMemcpyAsync(m->tok(), tokens_host, M * 4, cudaMemcpyHostToDevice, cs);
    if (e != cudaSuccess) return tfm::cuda_fail(e, "tokens host->device");
    st = tfm::forward_impl(m, m->tok(), B, S, m->logits(), m->sz.ldV, cs);
    if (st != TFM_OK) return st;
    e = tfm::copy_logits_to_host(m, logits_host, ld_logits, m->logits(), M, cs);
    if (e != cudaSuccess) return tfm::cuda_fail(e, "logits device->host");
    return TFM_OK;
}

tfm_status tfm_selftest_wait_timeout(int32_t limit_ms, void* stream) {
    if (limit_ms < 1 || limit_ms > 2000) return fail(TFM_EINVAL, "limit_ms must be in [1, 2000]");
    if (!tfm::device_error_word()) return fail(TFM_ECUDA, "device error word unavailable");
    const cudaError_t e = tfm::launch_selftest_wait((uint64_t)limit_ms * 1000000ull,
                                                    static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TFM_OK : tfm::cuda_fail(e, "self-test launch");
}

tfm_status tfm_profile_enable(void* handle, int32_t enable) {
    Model* m = static_cast<Model*>(handle);
    if (!m) return fail(TFM_EINVAL, "NULL handle");
    m->prof = enable != 0;
    return TFM_OK;
}

tfm_status tfm_profile_read(void* handle, double* ms, int64_t* launches) {
    Model* m = static_cast<Model*>(handle);
    if (!m || !ms || !launches) return fail(TFM_EINVAL, "NULL argument");
    for (const auto& r : m->runs) {
        const size_t n = r.kinds.size();
        cudaError_t e = cudaEventSynchronize(m->ev_pool[r.ev0 + n]);
        if (e != cudaSuccess) return tfm::cuda_fail(e, "profile event");
        for (size_t i = 0; i < n; ++i) {
            float t = 0.f;
            e = cudaEventElapsedTime(&t, m->ev_pool[r.ev0 + i], m->ev_pool[r.ev0 + i + 1]);
            if (e != cudaSuccess) return tfm::cuda_fail(e, "profile elapsed time");
            ms[r.kinds[i]] += t;
            launches[r.kinds[i]] += 1;
        }
    }
    m->runs.clear();
    m->ev_used = 0;
    return TFM_OK;
}

const char* tfm_profile_kind_name(int32_t kind) {
    static const char* names[TFM_PROFILE_KINDS] = {"embedding_rmsnorm", "rmsnorm", "qkv_rope_gemm",
                                                   "attention", "oproj_residual_gemm",
                                                   "gateup_swiglu_gemm", "down_residual_gemm",
                                                   "lmhead_gemm"};
    return (kind >= 0 && kind < TFM_PROFILE_KINDS) ? names[kind] : "";
}

tfm_status tfm_device_status(void* handle) {
    (void)handle;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return tfm::cuda_fail(e, "device synchronize");
    int* w = tfm::device_error_word();
    if (!w) return fail(TFM_ECUDA, "device error word unavailable");
    int v = 0, zero = 0;
    e = cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && v != 0) e = cudaMemcpy(w, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return tfm::cuda_fail(e, "read device error word");
    if (v == TFM_EBADTOKEN) return fail(TFM_EBADTOKEN, "a token id was outside [0, vocab)");
    if (v == TFM_ETIMEOUT) return fail(TFM_ETIMEOUT, "a pipeline wait timed out on the device");
    if (v != 0) return fail((tfm_status)v, "device error %d", v);
    return TFM_OK;
}

// ------------------------------------------------------------------ components

tfm_status tfm_embedding(const int32_t* tokens, const void* E, float* h, int64_t M, int32_t V,
                         int32_t D, int32_t mode, void* stream) {
    if (M < 0 || V < 1 || D < 1) return fail(TFM_EINVAL, "bad sizes");
    if (mode != TFM_FP32 && mode != TFM_BF16) return fail(TFM_EINVAL, "bad mode");
    if (D % (mode == TFM_BF16 ? 8 : 4)) return fail(TFM_EINVAL, "D must be a multiple of %d", mode == TFM_BF16 ? 8 : 4);
    if (M == 0) return TFM_OK;
    if (!tokens || !E || !h) return fail(TFM_EINVAL, "NULL pointer");
    if (!tfm::aligned16(E) || !tfm::aligned16(h)) return fail(TFM_EINVAL, "E and h must be 16-byte aligned");
    if (!tfm::aligned_to(tokens, 4)) return fail(TFM_EINVAL, "tokens must be 4-byte aligned");
    if (!tfm::device_error_word()) return fail(TFM_ECUDA, "device error word unavailable");
    cudaError_t e = tfm::launch_embedding(tokens, E, h, M, V, D, mode == TFM_BF16,
                                          static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TFM_OK : tfm::cuda_fail(e, "embedding launch");
}

tfm_status tfm_rmsnorm(const float* x, const float* g, void* y, int64_t M, int32_t D, float eps,
                       int32_t out_mode, void* stream) {
    if (M < 0 || D < 8 || D % 8) return fail(TFM_EINVAL, "D must be a positive multiple of 8");
    if (!(eps > 0.f)) return fail(TFM_EINVAL, "eps must be > 0");
    if (out_mode != TFM_FP32 && out_mode != TFM_BF16) return fail(TFM_EINVAL, "bad out_mode");
    if (M == 0) return TFM_OK;
    if (!x || !g || !y) return fail(TFM_EINVAL, "NULL pointer");
    if (!tfm::aligned16(x) || !tfm::aligned16(g) || !tfm::aligned16(y))
        return fail(TFM_EINVAL, "x, g, y must be 16-byte aligned");
    cudaError_t e = tfm::launch_rmsnorm(x, g, y, M, D, eps, out_mode == TFM_BF16,
                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TFM_OK : tfm::cuda_fail(e, "rmsnorm launch");
}

tfm_status tfm_rope(void* x, const int32_t* positions, int32_t B, int32_t H, int32_t S, int32_t dh,
                    float theta, int32_t mode, void* stream) {
    if (B < 0 || H < 0 || S < 0 || dh < 2 || dh % 2 || dh > 256) return fail(TFM_EINVAL, "bad sizes");
    if (!(theta > 1.f)) return fail(TFM_EINVAL, "theta must be > 1");
    if (mode != TFM_FP32 && mode != TFM_BF16) return fail(TFM_EINVAL, "bad mode");
    if ((int64_t)B * H * S == 0) return TFM_OK;
    if (!x) return fail(TFM_EINVAL, "NULL x");
    if (!tfm::aligned_to(x, mode == TFM_BF16 ? 2 : 4) || !tfm::aligned_to(positions, 4))
        return fail(TFM_EINVAL, "x must be aligned to its element size, positions to 4 bytes");
    cudaError_t e = tfm::launch_rope(x, positions, B, H, S, dh, theta, mode == TFM_BF16,
                                     static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TFM_OK : tfm::cuda_fail(e, "rope launch");
}

tfm_status tfm_causal_attention(const void* q, const void* k, const void* v, void* o, int32_t B,
                                int32_t H, int32_t Hkv, int32_t S, int32_t dh, float scale,
                                int32_t mode, void* stream) {
    return tfm_causal_attention_window(q, k, v, o, B, H, Hkv, S, dh, scale, 0, mode, stream);
}

tfm_status tfm_causal_attention_window(const void* q, const void* k, const void* v, void* o,
                                       int32_t B, int32_t H, int32_t Hkv, int32_t S, int32_t dh,
                                       float scale, int32_t window, int32_t mode, void* stream) {
    if (window < 0) return fail(TFM_EINVAL, "window must be >= 0");
    if (window >= S) window = 0;
    if (B < 0 || S < 0 || H < 1 || Hkv < 1 || H % Hkv) return fail(TFM_EINVAL, "bad head counts");
    if (mode != TFM_FP32 && mode != TFM_BF16) return fail(TFM_EINVAL, "bad mode");
    if (mode == TFM_BF16 && !tfm::attention_tc_supported(dh))
        return fail(TFM_EUNSUPPORTED, "bf16 attention: dh in {32,64,128}");
    if (mode == TFM_FP32 && (dh < 1 || dh > 128)) return fail(TFM_EUNSUPPORTED, "fp32 attention: dh <= 128");
    if (B == 0 || S == 0) return TFM_OK;
    if (!q || !k || !v || !o) return fail(TFM_EINVAL, "NULL pointer");
    if (!tfm::aligned16(q) || !tfm::aligned16(k) || !tfm::aligned16(v) || !tfm::aligned16(o))
        return fail(TFM_EINVAL, "q, k, v, o must be 16-byte aligned");
    if (scale <= 0.f) scale = 1.0f / std::sqrt((float)dh);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (mode == TFM_BF16) {
        tfm::AttnPlan plan;
        tfm_status ps = tfm::plan_attention_tc(&plan, q, k, v, o, B, H, Hkv, S, dh, scale);
        if (ps != TFM_OK) return fail(ps, "could not encode attention tensor maps");
        plan.window = window;
        e = tfm::launch_attention_tc(plan, cs);
    } else {
        e = tfm::launch_attention_simt(static_cast<const float*>(q), static_cast<const float*>(k),
                                       static_cast<const float*>(v), static_cast<float*>(o), B, H,
                                       Hkv, S, dh, scale, cs, window);
    }
    return e == cudaSuccess ? TFM_OK : tfm::cuda_fail(e, "attention launch");
}

size_t tfm_decode_attention_workspace_bytes(int32_t B, int32_t H, int32_t max_seq, int32_t dh) {
    if (B < 1 || H < 1 || max_seq < 1 || (dh != 32 && dh != 64 && dh != 128)) return 0;
    // the position word (256 bytes reserved), then the chunk partials
    return 256 + tfm::decode_partial_floats(B, H, max_seq, dh) * 4;
}

tfm_status tfm_decode_attention(const void* q, const void* k_cache, const void* v_cache, void* o,
                                int32_t B, int32_t H, int32_t Hkv, int32_t max_seq, int32_t pos,
                                int32_t dh, float scale, int32_t window, void* workspace,
                                size_t workspace_bytes, void* stream) {
    if (B < 0 || H < 1 || Hkv < 1 || H % Hkv || max_seq < 1) return fail(TFM_EINVAL, "bad sizes");
    if (pos < 0 || pos >= max_seq) return fail(TFM_EINVAL, "pos=%d outside [0, max_seq=%d)", pos, max_seq);
    if (window < 0) return fail(TFM_EINVAL, "window must be >= 0");
    if (!tfm::decode_supported(dh, H / Hkv))
        return fail(TFM_EUNSUPPORTED, "dh in {32, 64, 128}, H/Hkv in {1, 2, 4, 8, 16} (<= 8 at dh 128)");
    if (B == 0) return TFM_OK;
    if (!q || !k_cache || !v_cache || !o || !workspace) return fail(TFM_EINVAL, "NULL pointer");
    if (!tfm::aligned16(q) || !tfm::aligned16(k_cache) || !tfm::aligned16(v_cache) ||
        !tfm::aligned16(o) || !tfm::aligned16(workspace))
        return fail(TFM_EINVAL, "pointers must be 16-byte aligned");
    if (workspace_bytes < tfm_decode_attention_workspace_bytes(B, H, max_seq, dh))
        return fail(TFM_EINVAL, "workspace too small");
    if (scale <= 0.f) scale = 1.0f / std::sqrt((float)dh);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // The position is copied from the host at call time, which a recorded graph
    // could not replay with a new value: refuse a capturing stream up front
    // instead of letting the capture fail.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(cs, &cap) == cudaSuccess && cap == cudaStreamCaptureStatusActive)
        return fail(TFM_EINVAL, "tfm_decode_attention cannot be recorded into a graph (the position "
                                "is copied from the host at call time); use tfm_decode_step");
    int* pos_dev = static_cast<int*>(workspace);
    float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + 256);
    // The kernel reads the position (and prefetches cache rows) before its grid
    // dependency wait, so the position must not come from the kernel launched just
    // before it: a stream-ordered copy has no programmatic early start.
    cudaError_t e = cudaMemcpyAsync(pos_dev, &pos, sizeof(int), cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess)
        e = tfm::launch_decode_attention(q, k_cache, v_cache, part, o, B, H, Hkv, max_seq, pos_dev,
                                         dh, scale, cs, window);
    return e == cudaSuccess ? TFM_OK : tfm::cuda_fail(e, "decode attention launch");
}

tfm_status tfm_linear(const void* x, const void* W, void* y, int64_t M, int32_t N, int32_t K,
                      int64_t ldy, int32_t out_fp32, int32_t accumulate, int32_t mode, void* stream) {
    if (M < 0 || M > INT32_MAX || N < 1 || K < 1 || ldy < N || ldy % 8) return fail(TFM_EINVAL, "bad sizes");
    if (mode != TFM_FP32 && mode != TFM_BF16) return fail(TFM_EINVAL, "bad mode");
    if (!out_fp32 && (accumulate || mode != TFM_BF16)) return fail(TFM_EINVAL, "bf16 output: bf16 mode, no accumulate");
    if (mode == TFM_BF16 && K % 8) return fail(TFM_EINVAL, "bf16 mode: K %% 8 == 0");
    if (M == 0) return TFM_OK;
    if (!x || !W || !y) return fail(TFM_EINVAL, "NULL pointer");
    if (!tfm::aligned16(x) || !tfm::aligned16(W) || !tfm::aligned16(y)) return fail(TFM_EINVAL, "pointers must be 16-byte aligned");
    const int kind = out_fp32 ? (accumulate ? tfm::EPI_ACCUM_F32 : tfm::EPI_STORE_F32) : tfm::EPI_STORE_BF16;
    tfm::EpiParams epi = tfm::epi_basic(kind, (int)M, N, y, ldy);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (mode == TFM_BF16) {
        tfm::GemmPlan plan;
        tfm_status st = tfm::plan_gemm_tc(&plan, x, K, W, nullptr, K, (int)M, N, K, epi);
        if (st != TFM_OK) return fail(st, "tensor map encoding failed");
        e = tfm::launch_gemm_tc(plan, cs);
    } else {
        e = tfm::launch_gemm_simt(static_cast<const float*>(x), static_cast<const float*>(W), nullptr,
                                  (int)M, N, K, epi, cs);
    }
    return e == cudaSuccess ? TFM_OK : tfm::cuda_fail(e, "linear launch");
}

size_t tfm_swiglu_workspace_bytes(int64_t M, int32_t F, int32_t mode) {
    if (M < 0 || F < 1) return 0;
    return (size_t)M * F * (mode == TFM_BF16 ? 2 : 4);
}

tfm_status tfm_swiglu(const void* x, const void* w1, const void* w3, const void* w2, float* y,
                      int64_t M, int32_t D, int32_t F, int32_t accumulate, void* workspace,
                      size_t workspace_bytes, int32_t mode, void* stream) {
    if (M < 0 || M > INT32_MAX || D < 1 || F < 1) return fail(TFM_EINVAL, "bad sizes");
    if (mode != TFM_FP32 && mode != TFM_BF16) return fail(TFM_EINVAL, "bad mode");
    if (D % 8 || F % 8) return fail(TFM_EINVAL, "D and F must be multiples of 8");
    if (M == 0) return TFM_OK;
    if (!x || !w1 || !w3 || !w2 || !y || !workspace) return fail(TFM_EINVAL, "NULL pointer");
    if (workspace_bytes < tfm_swiglu_workspace_bytes(M, F, mode)) return fail(TFM_EINVAL, "workspace too small");
    if (!tfm::aligned16(x) || !tfm::aligned16(w1) || !tfm::aligned16(w3) || !tfm::aligned16(w2) ||
        !tfm::aligned16(y) || !tfm::aligned16(workspace))
        return fail(TFM_EINVAL, "pointers must be 16-byte aligned");
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    tfm::EpiParams eg = tfm::epi_basic(tfm::EPI_SWIGLU, (int)M, F, workspace, F);
    tfm::EpiParams ed = tfm::epi_basic(accumulate ? tfm::EPI_ACCUM_F32 : tfm::EPI_STORE_F32, (int)M,
                                       D, y, D);
    cudaError_t e;
    if (mode == TFM_BF16) {
        eg.out_bf16 = 1;
        tfm::GemmPlan pg, pd;
        tfm_status st = tfm::plan_gemm_tc(&pg, x, D, w1, w3, D, (int)M, F, D, eg);
        if (st == TFM_OK) st = tfm::plan_gemm_tc(&pd, workspace, F, w2, nullptr, F, (int)M, D, F, ed);
        if (st != TFM_OK) return fail(st, "tensor map encoding failed");
        e = tfm::launch_gemm_tc(pg, cs);
        if (e == cudaSuccess) e = tfm::launch_gemm_tc(pd, cs);
    } else {
        eg.out_bf16 = 0;
        e = tfm::launch_gemm_simt(static_cast<const float*>(x), static_cast<const float*>(w1),
                                  static_cast<const float*>(w3), (int)M, F, D, eg, cs);
        if (e == cudaSuccess)
            e = tfm::launch_gemm_simt(static_cast<const float*>(workspace),
                                      static_cast<const float*>(w2), nullptr, (int)M, D, F, ed, cs);
    }
    return e == cudaSuccess ? TFM_OK : tfm::cuda_fail(e, "swiglu launch");
}

}  // extern "C"
