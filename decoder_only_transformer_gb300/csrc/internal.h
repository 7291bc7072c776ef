// internal.h - declarations shared by libtfm's translation units (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tfm.h"

namespace tfm {

// Epilogues a GEMM applies to its fp32 accumulator tile.
enum EpiKind {
    EPI_STORE_F32 = 0,   // out[m, n] = acc                      (fp32, e.g. logits)
    EPI_ACCUM_F32 = 1,   // out[m, n] += acc                     (fp32 residual stream)
    EPI_STORE_BF16 = 2,  // out[m, n] = bf16(acc)
    EPI_SWIGLU = 3,      // out[m, f] = silu(gate) * up          (bf16 or fp32 hidden activation)
    EPI_QKV_ROPE = 4,    // RoPE on q/k columns, scatter to head-major q, k, v
    EPI_LSE = 5,         // no output: per row running (max, sum exp) of the tile's
                         // columns and the target column's logit (fused cross-entropy)
    EPI_GELU = 6,        // out[m, n] = gelu(acc), exact form  (bf16 or fp32 hidden activation)
};

struct EpiParams {
    int kind;
    int M, N;             // output rows; output columns (F for EPI_SWIGLU, Dq+2Dkv for QKV)
    void* out;            // STORE/ACCUM/SWIGLU destination
    int64_t ldo;          // its row stride in elements
    int out_bf16;         // SWIGLU/QKV: 1 = bf16 outputs, 0 = fp32
    // EPI_QKV_ROPE: row m = b*S + s; columns [0,Dq) -> q[b,h,s,:], then k, then v;
    // q and k are rotated for position pos0 + s (pos0 = 0 for a whole sequence, the
    // cache length for a decode step)
    int S, n_head, n_kv_head, dh;
    int pos0;
    // k and v into a KV cache instead: [B, n_kv_head, kv_stride, dh] at position
    // pos0 + s (0: head-major like q, [B, n_kv_head, S, dh])
    int kv_stride;
    // when set, pos0 is read from this device word (a decode step replayed from a
    // recorded graph, the position changing between replays)
    const int* pos0_dev;
    const float* rope_cs;    // [>= S, dh/2, 2]: cos, sin of s * theta^(-2i/dh); null: no rotation
    // fp32 [N], added to the accumulator column before everything else (the
    // biased linears of the GPT-2-style family); null: none
    const float* bias;
    void* q;
    void* k;
    void* v;
    // Tensor-core GEMM: 1 = each staged 32 x 32 output block is written by one TMA
    // store (or reduce-add for EPI_ACCUM_F32) through the output maps of TcMaps.
    int tma_out;
    // EPI_LSE: targets [M]; lse_part [M][lse_slots] (max, sum of exp(z - max))
    // pairs, slot 2 * column tile + half (the two warps of a lane quarter take
    // alternate 32-column chunks); lse_tgt [M] the logit of the target column.
    const int32_t* targets;
    float2* lse_part;
    float* lse_tgt;
    int lse_slots;
};

// Launch with programmatic stream serialization allowed (see pdl_wait in
// common.cuh): only for kernels that call pdl_wait() before global accesses.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same with a cluster of two CTAs along x (CTA pairs for cta_group::2).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_pair(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                   cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Library-global device error word of the current device (see raise_error).
int* device_error_word();
// Sets the thread-local text tfm_last_error() returns.
void set_last_error(const char* msg);
int sm_count();
const char* cuda_error_text(cudaError_t e);

// ---- elementwise kernels (k_rows.cu)
// How a row is normalised: RMSNorm (the default), LayerNorm with shift b, or no
// norm (cast only).  h_out: also store the fp32 normalised row (may equal the
// input).  pos (embedding kernels only): position rows [>= S, D] in the
// embedding's type added to E[tok[m]], row m taking position m % S, plus
// *pos_dev when set (a decode step's position, read on the device).
enum NormKind { kNormRms = 0, kNormLayer = 1, kNormNone = 2 };
struct NormArgs {
    int kind;
    const float* b;
    float* h_out;
    const void* pos;
    int S;
    const int* pos_dev;
};
cudaError_t launch_embedding(const int32_t* tok, const void* E, float* h, int64_t M, int V,
                             int D, int e_bf16, cudaStream_t st);
// g_static = 1: no launch on the stream writes g (a model's gain), so a few-row
// launch may load it before its grid dependency wait.
cudaError_t launch_rmsnorm(const float* x, const float* g, void* y, int64_t M, int D, float eps,
                           int out_bf16, cudaStream_t st, int g_static = 0,
                           const NormArgs* na = nullptr);
cudaError_t launch_rope(void* x, const int32_t* pos, int B, int H, int S, int dh, float theta,
                        int is_bf16, cudaStream_t st);
cudaError_t launch_selftest_wait(uint64_t limit_ns, cudaStream_t st);
// h = E[tok] and y = RMSNorm(h) * g in one pass (bf16: E and y bf16; else fp32).
cudaError_t launch_embed_rmsnorm(const int32_t* tok, const void* E, const float* g, float* h,
                                 void* y, int64_t M, int V, int D, float eps, int bf16,
                                 cudaStream_t st, int g_static = 0, const NormArgs* na = nullptr);

// ---- fused cross-entropy (k_loss.cu): per row of materialised logits [M, ld]
// one (max, sum exp) slot and the target logit; then, from any number of slots
// per row, lse = max + log(sum), loss = lse - target logit (NaN and
// TFM_EBADTOKEN for a target outside [0, V)); mean over the M rows in a fixed
// order (one CTA).  loss_out / lse_out may be null; mean_out may be null.
cudaError_t launch_lse_rows(const float* logits, int64_t ld, int M, int V, const int32_t* targets,
                            float2* part, float* tgt, cudaStream_t st);
cudaError_t launch_lse_finish(const float2* part, int slots, const float* tgt,
                              const int32_t* targets, int M, int V, float* loss_out,
                              float* lse_out, float* loss_tmp, float* mean_out, cudaStream_t st);

// ---- CUDA-core kernels (k_simt.cu), fp32 mode
// C = A[M,K] . B[N,K]^T (and A . B2^T for EPI_SWIGLU), then the epilogue.
cudaError_t launch_gemm_simt(const float* A, const float* B, const float* B2, int M, int N,
                             int K, const EpiParams& epi, cudaStream_t st);
cudaError_t launch_attention_simt(const float* q, const float* k, const float* v, float* o,
                                  int B, int H, int Hkv, int S, int dh, float scale,
                                  cudaStream_t st, int window = 0);

// ---- tensor-core GEMM (k_gemm_tc.cu), bf16 mode
// Tensor maps of one GEMM: A [M,K] and B [N,K] bf16 row-major (B2 = W3 for SwiGLU).
struct TcMaps {
    CUtensorMap a;
    CUtensorMap b;
    CUtensorMap b2;
    // Output maps when EpiParams::tma_out is set, box 32 x 32: `out` ([M, N] fp32
    // or bf16) for the plain, residual and SwiGLU kinds; `oq`, `ok`, `ov`
    // ([B*heads, S, dh] bf16) for the QKV kind.
    CUtensorMap out;
    CUtensorMap oq;
    CUtensorMap ok;
    CUtensorMap ov;
};
struct GemmPlan {
    TcMaps maps;
    int M, N, K;          // N = GEMM columns covered by tiles (F for SwiGLU)
    int block_n;          // tile width (128 or 256); SwiGLU: gate+up halves of block_n/2
    int dual;             // SwiGLU: B tile = [W1 rows; W3 rows]
    int pair;             // 1: CTA pairs (cta_group::2) on 256-row tiles
    int n_fast;           // tile order: 1 = column blocks fastest, 0 = row blocks fastest
    // M <= 128: the weight-streaming kernel (k_gemm_skinny.cu): A rows padded to
    // sk_nm, sk_tiles tiles of 128 W rows (64 per weight for SwiGLU), K split
    // over sk_splits CTAs of a cluster.  maps.a boxes sk_nm rows of A; maps.b
    // (and maps.b2) box the W rows of a tile.
    int skinny, sk_nm, sk_tiles, sk_splits;
    // 1: no launch on the stream writes B (a model weight), so its loads may
    // start before the grid dependency wait (set by the model's own plans)
    int b_static;
    EpiParams epi;
    // Weight-streaming plans with sk_nm == 16: when norm_x is set, A is the
    // RMSNorm of the fp32 rows norm_x [M, K] with gain norm_g [K] (bf16 of
    // x / sqrt(mean(x^2) + eps) * g), computed by the kernel in place of loading
    // A; null: A as given.
    const float* norm_x;
    const float* norm_g;
    float norm_eps;
};
// Builds the tensor maps; returns TFM_OK or an error status with a message.
tfm_status plan_gemm_tc(GemmPlan* plan, const void* A, int64_t lda, const void* B,
                        const void* B2, int64_t ldb, int M, int N, int K, const EpiParams& epi);
cudaError_t launch_gemm_tc(const GemmPlan& plan, cudaStream_t st);
cudaError_t launch_gemm_skinny(const GemmPlan& plan, cudaStream_t st);

// ---- attention of one new query per sequence over a KV cache (k_decode.cu):
// q [B, H, dh], caches [B, Hkv, max_seq, dh] (positions [0, L) read), o [B, H*dh]
// bf16; part holds decode_partial_floats(B, H, max_seq, dh) floats of scratch.
// The attended length is *pos_dev + 1 (read on the device, so the launch can be
// replayed from a recorded graph at every position); the grid covers max_seq.
size_t decode_partial_floats(int B, int H, int max_seq, int dh);
bool decode_supported(int dh, int group);
// window > 0: only keys [pos - window + 1, pos] (a sliding-window layer).
cudaError_t launch_decode_attention(const void* q, const void* kc, const void* vc, float* part,
                                    void* o, int B, int H, int Hkv, int max_seq,
                                    const int* pos_dev, int dh, float scale, cudaStream_t st,
                                    int window = 0);
// Stores the decode step's position and copies its B tokens into device words.
cudaError_t launch_decode_setup(int* pos_dev, int pos, const int32_t* tok, int32_t* tok_dev, int B,
                                cudaStream_t st);

// ---- bf16 flash attention on tcgen05 (k_attention_tc.cu, k_attention_pp.cu,
// k_attention_short.cu), dh in {32, 64, 128}
struct AttnPlan {
    CUtensorMap qmap, kmap, vmap;   // [B*heads, S, dh] views of q, k, v
    int B, H, Hkv, S, dh;
    float scale;
    void* o;                        // [B, S, H*dh] bf16
    int window;                     // > 0: sliding window (query i sees keys i-window < j <= i)
};
bool attention_tc_supported(int dh);
tfm_status plan_attention_tc(AttnPlan* p, const void* q, const void* k, const void* v, void* o,
                             int B, int H, int Hkv, int S, int dh, float scale);
cudaError_t launch_attention_tc(const AttnPlan& p, cudaStream_t st);
// two query tiles per CTA, dh in {32, 64} (k_attention_pp.cu)
cudaError_t launch_attention_pp(const AttnPlan& p, cudaStream_t st);
// dh 32, S <= 256, no window: the three causal 128 x 128 blocks of a (sequence,
// head) side by side (k_attention_short.cu)
bool attention_short_supported(int dh, int S, int window);
cudaError_t launch_attention_short(const AttnPlan& p, cudaStream_t st);

}  // namespace tfm
