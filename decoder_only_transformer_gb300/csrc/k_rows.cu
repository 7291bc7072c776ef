// k_rows.cu - HBM-bound row kernels: embedding gather, RMSNorm (fp32 in,
// bf16/fp32 out) and the standalone RoPE used by the component entry point.
//
// All three move each byte once: 16-byte vector loads and stores, one warp per
// row, the row held in registers between the reduction and the write.
#include "common.cuh"
#include "internal.h"

namespace tfm {

// ------------------------------------------------------------------ embedding
// h[m, :] = E[tok[m], :] (CS336 walkthrough, section 5.2: the Embedding layer
// looks each token id up in a [vocab, d_model] table).  One warp per row; an
// id outside [0, V) writes zeros and raises TFM_EBADTOKEN.
template <bool kBf16>
__global__ void __launch_bounds__(256) k_embedding(const int32_t* __restrict__ tok,
                                                   const void* __restrict__ E,
                                                   float* __restrict__ h, int64_t M, int V, int D,
                                                   int* err) {
    const int lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t m = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); m < M;
         m += warps) {
        const int t = __ldg(tok + m);
        float* dst = h + m * D;
        const bool ok = (t >= 0 && t < V);
        if (!ok && lane == 0) raise_error(err, TFM_EBADTOKEN);
        if (kBf16) {
            const uint4* src = reinterpret_cast<const uint4*>(
                static_cast<const __nv_bfloat16*>(E) + (int64_t)(ok ? t : 0) * D);
            for (int c = lane; c < D / 8; c += 32) {
                uint4 w = ok ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
                float4 lo = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
                float4 hi = make_float4(bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w));
                reinterpret_cast<float4*>(dst)[2 * c] = lo;
                reinterpret_cast<float4*>(dst)[2 * c + 1] = hi;
            }
        } else {
            const float4* src = reinterpret_cast<const float4*>(
                static_cast<const float*>(E) + (int64_t)(ok ? t : 0) * D);
            for (int c = lane; c < D / 4; c += 32)
                reinterpret_cast<float4*>(dst)[c] = ok ? __ldg(src + c) : make_float4(0, 0, 0, 0);
        }
    }
}

cudaError_t launch_embedding(const int32_t* tok, const void* E, float* h, int64_t M, int V, int D,
                             int e_bf16, cudaStream_t st) {
    if (M <= 0) return cudaSuccess;
    int64_t blocks = (M + 7) / 8;
    const int cap = sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (e_bf16)
        return launch_pdl(k_embedding<true>, dim3((unsigned)blocks), dim3(256), 0, st, tok, E, h, M,
                          V, D, device_error_word());
    return launch_pdl(k_embedding<false>, dim3((unsigned)blocks), dim3(256), 0, st, tok, E, h, M, V,
                      D, device_error_word());
}

// ------------------------------------------------------------------ norms
// Every norm below works on fp32 rows and rounds once to the output type
// (CS336 walkthrough, section 5.6: fp32 through the gain multiply, then cast):
//   RMSNorm    y = x / sqrt(mean(x^2) + eps) * g          (section 5.6)
//   LayerNorm  y = (x - mean) / sqrt(var + eps) * g + b    (population variance;
//              "Chapter 4", section 5, the GPT-2-style family)
//   none       y = x                                       (the input of a
//              post-norm block's first projections, cast only)
// NormArgs::h_out also stores the fp32 normalised row (post-norm blocks
// normalise the residual stream itself; it may be x: each element is read
// before it is written, by the same thread).  The embedding kernels add the
// position row of token m (m % S) to E[tok[m]] when NormArgs::pos is set.

// Output of one 4-float group: a = norm(v) (the mean already taken out of v
// for LayerNorm), then the optional fp32 copy and the store.
template <int kKind, bool kBf16Y>
__device__ __forceinline__ void norm_store(const float4 v, float r, const float4* g4,
                                           const float4* b4, int c, float* hrow, void* yrow) {
    float4 a = v;
    if (kKind != kNormNone) {
        const float4 w = __ldg(g4 + c);
        a = make_float4(v.x * r * w.x, v.y * r * w.y, v.z * r * w.z, v.w * r * w.w);
        if (kKind == kNormLayer) {
            const float4 bb = __ldg(b4 + c);
            a.x += bb.x; a.y += bb.y; a.z += bb.z; a.w += bb.w;
        }
    }
    if (kKind != kNormRms && hrow) reinterpret_cast<float4*>(hrow)[c] = a;
    if (kBf16Y) {
        uint2 o;
        o.x = pack_bf16x2(a.x, a.y);
        o.y = pack_bf16x2(a.z, a.w);
        reinterpret_cast<uint2*>(yrow)[c] = o;
    } else {
        reinterpret_cast<float4*>(yrow)[c] = a;
    }
}

__device__ __forceinline__ float sum4(const float4 v) { return v.x + v.y + v.z + v.w; }
__device__ __forceinline__ float sq4(const float4 v) {
    return v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
}
__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

// The scale r of a row held as kV groups per lane (groups c >= n4 are zero):
// for LayerNorm the mean is subtracted from the groups in range first.
template <int kKind, int kV>
__device__ __forceinline__ float warp_norm_scale(float4 (&v)[kV], int lane, int n4, int D,
                                                 float eps) {
    if (kKind == kNormNone) return 1.f;
    if (kKind == kNormLayer) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < kV; ++i) s += sum4(v[i]);
        const float mu = warp_sum(s) / (float)D;
#pragma unroll
        for (int i = 0; i < kV; ++i)
            if (lane + 32 * i < n4) {
                v[i].x -= mu; v[i].y -= mu; v[i].z -= mu; v[i].w -= mu;
            }
    }
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kV; ++i) ss += sq4(v[i]);
    return 1.0f / sqrtf(warp_sum(ss) / (float)D + eps);
}

// Group c of the row of E[t] (+ position row), 4 floats.
template <bool kBf16E>
__device__ __forceinline__ float4 load_group(const void* base, int64_t row, int D, int c) {
    if (kBf16E) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(
                                  static_cast<const __nv_bfloat16*>(base) + row * D) + c);
        return make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
    }
    return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + row * D) + c);
}

// ------------------------------------------------------------------ embedding + first norm
// The forward's first steps in one pass: h[m] = E[tok[m]] (+ the position row)
// in fp32 (the residual stream) and y[m] = norm(h[m]) (the first block's input
// norm), the row held in registers in between.  One warp per row; lane l owns
// the 4-float groups l, l+32, ...; an id outside [0, V) writes zeros and raises
// TFM_EBADTOKEN.
template <int kKind, int kV, bool kBf16E, bool kBf16Y>
__global__ void __launch_bounds__(256, kV == 16 ? 3 : 1) k_embed_rmsnorm(const int32_t* __restrict__ tok,
                                                       const void* __restrict__ E,
                                                       const float* __restrict__ g,
                                                       float* __restrict__ h, void* __restrict__ y,
                                                       int64_t M, int V, int D, float eps,
                                                       NormArgs na, int* err) {
    const int lane = threadIdx.x & 31;
    // The gain, staged once per CTA: each warp's stores then wait on no global
    // load after its row's reduction.  With that and three CTAs per SM (rows of
    // 1025 to 2048 floats, 64 per lane, in 80 registers), 24 rows are in flight
    // per SM instead of 16: the GQA workload's gather + norm 52.1 -> 38.4 us, the
    // long-context one's 21.0 -> 18.6 us (each warp's row is a chain of dependent
    // memory waits).  Longer rows (128 floats per lane) do not fit that register
    // budget and take no occupancy bound.
    __shared__ float4 gs[kKind == kNormRms ? kV * 32 : 1];
    pdl_wait();
    pdl_trigger();
    const int n4 = D >> 2;
    if (kKind == kNormRms) {
        for (int c = threadIdx.x; c < n4; c += blockDim.x) gs[c] = __ldg(reinterpret_cast<const float4*>(g) + c);
        __syncthreads();
    }
    const int64_t m = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (m >= M) return;
    const int t = __ldg(tok + m);
    const bool ok = (t >= 0 && t < V);
    if (!ok && lane == 0) raise_error(err, TFM_EBADTOKEN);
    const int64_t row = ok ? t : 0;
    const int64_t prow = na.pos ? (na.pos_dev ? __ldg(na.pos_dev) : 0) + m % na.S : 0;
    float4 v[kV];
#pragma unroll
    for (int i = 0; i < kV; ++i) {
        const int c = lane + 32 * i;
        v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < n4 && ok) v[i] = load_group<kBf16E>(E, row, D, c);
        if (c < n4 && na.pos) {
            const float4 p = load_group<kBf16E>(na.pos, prow, D, c);
            v[i].x += p.x; v[i].y += p.y; v[i].z += p.z; v[i].w += p.w;
        }
        if (c < n4) reinterpret_cast<float4*>(h + m * D)[c] = v[i];
    }
    const float r = warp_norm_scale<kKind, kV>(v, lane, n4, D, eps);
    const float4* g4 = reinterpret_cast<const float4*>(g);
    const float4* b4 = reinterpret_cast<const float4*>(na.b);
    void* yrow = kBf16Y ? (void*)(static_cast<__nv_bfloat16*>(y) + m * D)
                        : (void*)(static_cast<float*>(y) + m * D);
    if (kKind == kNormRms && kBf16Y) {
#pragma unroll
        for (int i = 0; i < kV; ++i) {
            const int c = lane + 32 * i;
            if (c >= n4) break;
            const float4 w = gs[c];
            uint2 o;
            o.x = pack_bf16x2(v[i].x * r * w.x, v[i].y * r * w.y);
            o.y = pack_bf16x2(v[i].z * r * w.z, v[i].w * r * w.w);
            reinterpret_cast<uint2*>(yrow)[c] = o;
        }
        return;
    }
#pragma unroll
    for (int i = 0; i < kV; ++i) {
        const int c = lane + 32 * i;
        if (c >= n4) break;
        norm_store<kKind, kBf16Y>(v[i], r, g4, b4, c, nullptr, yrow);
    }
}

// ------------------------------------------------------------------ few rows
// For a handful of rows (a decode step has one per sequence) the warp-per-row
// kernels leave the latency of each dependent load exposed.  Here one CTA of 256
// threads takes a row: thread t owns the 4-float groups t, t + 256, ... (kPer of
// them); a model's gain is a weight that no launch writes, so it is loaded
// before the dependency wait (g_static); the sums are reduced over the block.
// kEmbed: the row is E[tok[m]] (+ position row), also written to h, as in
// k_embed_rmsnorm.
constexpr int kRowKernelMaxM = 64;

__device__ __forceinline__ float block_sum(float s, float* red, int tid) {
    s = warp_sum(s);
    __syncthreads();                                  // red may hold the previous sum
    if ((tid & 31) == 0) red[tid >> 5] = s;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += red[w];
    return t;
}

template <int kKind, int kPer, bool kEmbed, bool kBf16E, bool kBf16Y>
__global__ void __launch_bounds__(256) k_norm_row(const int32_t* __restrict__ tok,
                                                  const void* __restrict__ X,
                                                  const float* __restrict__ g,
                                                  float* __restrict__ h, void* __restrict__ y,
                                                  int V, int D, float eps, int g_static,
                                                  NormArgs na, int* err) {
    __shared__ float red[8];
    const int tid = threadIdx.x;
    const int64_t m = blockIdx.x;
    const int n4 = D >> 2;
    const float4* g4 = reinterpret_cast<const float4*>(g);
    float4 gv[kPer];
    if (!g_static) pdl_wait();                   // g may come from the launch before
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int c = tid + 256 * i;
        gv[i] = (c < n4 && kKind != kNormNone) ? __ldg(g4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    pdl_wait();
    pdl_trigger();
    int64_t row = m;
    bool ok = true;
    if (kEmbed) {
        const int t = __ldg(tok + m);
        ok = (t >= 0 && t < V);
        if (!ok && tid == 0) raise_error(err, TFM_EBADTOKEN);
        row = ok ? t : 0;
    }
    const int64_t prow = na.pos ? (na.pos_dev ? __ldg(na.pos_dev) : 0) + m % na.S : 0;
    float4 v[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int c = tid + 256 * i;
        v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < n4 && ok) v[i] = load_group<kBf16E>(X, row, D, c);
        if (kEmbed && c < n4 && na.pos) {
            const float4 p = load_group<kBf16E>(na.pos, prow, D, c);
            v[i].x += p.x; v[i].y += p.y; v[i].z += p.z; v[i].w += p.w;
        }
        if (kEmbed && c < n4) reinterpret_cast<float4*>(h + m * D)[c] = v[i];
    }
    float r = 1.f;
    if (kKind != kNormNone) {
        if (kKind == kNormLayer) {
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < kPer; ++i) s += sum4(v[i]);
            const float mu = block_sum(s, red, tid) / (float)D;
#pragma unroll
            for (int i = 0; i < kPer; ++i)
                if (tid + 256 * i < n4) {
                    v[i].x -= mu; v[i].y -= mu; v[i].z -= mu; v[i].w -= mu;
                }
        }
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < kPer; ++i) ss += sq4(v[i]);
        r = 1.0f / sqrtf(block_sum(ss, red, tid) / (float)D + eps);
    }
    const float4* b4 = reinterpret_cast<const float4*>(na.b);
    void* yrow = kBf16Y ? (void*)(static_cast<__nv_bfloat16*>(y) + m * D)
                        : (void*)(static_cast<float*>(y) + m * D);
    float* hrow = na.h_out ? na.h_out + m * D : nullptr;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int c = tid + 256 * i;
        if (c >= n4) continue;
        float4 a = v[i];
        if (kKind != kNormNone) {
            const float4 w = gv[i];
            a = make_float4(v[i].x * r * w.x, v[i].y * r * w.y, v[i].z * r * w.z, v[i].w * r * w.w);
            if (kKind == kNormLayer) {
                const float4 bb = __ldg(b4 + c);
                a.x += bb.x; a.y += bb.y; a.z += bb.z; a.w += bb.w;
            }
        }
        if (kKind != kNormRms && hrow) reinterpret_cast<float4*>(hrow)[c] = a;
        if (kBf16Y) {
            uint2 o;
            o.x = pack_bf16x2(a.x, a.y);
            o.y = pack_bf16x2(a.z, a.w);
            reinterpret_cast<uint2*>(yrow)[c] = o;
        } else {
            reinterpret_cast<float4*>(yrow)[c] = a;
        }
    }
}

// Few-row launch (M <= kRowKernelMaxM, D <= 8192); returns false when it does not apply.
template <bool kEmbed>
static bool norm_row_launch(cudaError_t* e, const int32_t* tok, const void* X, const float* g,
                            float* h, void* y, int64_t M, int V, int D, float eps, int bf16,
                            int g_static, const NormArgs& na, cudaStream_t st) {
    if (M > kRowKernelMaxM || D > 8192) return false;
    const int per = (D / 4 + 255) / 256;
    const dim3 grid((unsigned)M), block(256);
    int* err = device_error_word();
#define TFM_ROW_LAUNCH(K, P)                                                                     \
    *e = bf16 ? launch_pdl(k_norm_row<K, P, kEmbed, kEmbed, true>, grid, block, 0, st, tok, X, g, \
                           h, y, V, D, eps, g_static, na, err)                                     \
              : launch_pdl(k_norm_row<K, P, kEmbed, false, false>, grid, block, 0, st, tok, X, g, \
                           h, y, V, D, eps, g_static, na, err)
#define TFM_ROW_KIND(K)                      \
    if (per <= 1) TFM_ROW_LAUNCH(K, 1);      \
    else if (per <= 2) TFM_ROW_LAUNCH(K, 2); \
    else if (per <= 4) TFM_ROW_LAUNCH(K, 4); \
    else TFM_ROW_LAUNCH(K, 8);
    if (na.kind == kNormLayer) {
        TFM_ROW_KIND(kNormLayer)
    } else if (na.kind == kNormNone) {
        TFM_ROW_KIND(kNormNone)
    } else {
        TFM_ROW_KIND(kNormRms)
    }
#undef TFM_ROW_KIND
#undef TFM_ROW_LAUNCH
    return true;
}

template <int kKind, int kV>
cudaError_t embed_norm_kind(const int32_t* tok, const void* E, const float* g, float* h, void* y,
                            int64_t M, int V, int D, float eps, int bf16, const NormArgs& na,
                            cudaStream_t st) {
    const dim3 blocks((unsigned)((M + 7) / 8));
    if (bf16)
        return launch_pdl(k_embed_rmsnorm<kKind, kV, true, true>, blocks, dim3(256), 0, st, tok, E,
                          g, h, y, M, V, D, eps, na, device_error_word());
    return launch_pdl(k_embed_rmsnorm<kKind, kV, false, false>, blocks, dim3(256), 0, st, tok, E, g,
                      h, y, M, V, D, eps, na, device_error_word());
}

template <int kV>
cudaError_t embed_norm_launch(const int32_t* tok, const void* E, const float* g, float* h, void* y,
                              int64_t M, int V, int D, float eps, int bf16, const NormArgs& na,
                              cudaStream_t st) {
    if (na.kind == kNormLayer)
        return embed_norm_kind<kNormLayer, kV>(tok, E, g, h, y, M, V, D, eps, bf16, na, st);
    if (na.kind == kNormNone)
        return embed_norm_kind<kNormNone, kV>(tok, E, g, h, y, M, V, D, eps, bf16, na, st);
    return embed_norm_kind<kNormRms, kV>(tok, E, g, h, y, M, V, D, eps, bf16, na, st);
}

cudaError_t launch_embed_rmsnorm(const int32_t* tok, const void* E, const float* g, float* h,
                                 void* y, int64_t M, int V, int D, float eps, int bf16,
                                 cudaStream_t st, int g_static, const NormArgs* nap) {
    if (M <= 0) return cudaSuccess;
    const NormArgs na = nap ? *nap : NormArgs{};
    cudaError_t e;
    if (norm_row_launch<true>(&e, tok, E, g, h, y, M, V, D, eps, bf16, g_static, na, st)) return e;
    const int groups = (D / 4 + 31) / 32;   // 4-float groups per lane
    if (groups <= 1) return embed_norm_launch<1>(tok, E, g, h, y, M, V, D, eps, bf16, na, st);
    if (groups <= 2) return embed_norm_launch<2>(tok, E, g, h, y, M, V, D, eps, bf16, na, st);
    if (groups <= 4) return embed_norm_launch<4>(tok, E, g, h, y, M, V, D, eps, bf16, na, st);
    if (groups <= 8) return embed_norm_launch<8>(tok, E, g, h, y, M, V, D, eps, bf16, na, st);
    if (groups <= 16) return embed_norm_launch<16>(tok, E, g, h, y, M, V, D, eps, bf16, na, st);
    if (groups <= 32) return embed_norm_launch<32>(tok, E, g, h, y, M, V, D, eps, bf16, na, st);
    // Rows beyond 4096: the gather (with the position rows) and the norm as two launches.
    if (na.pos) return cudaErrorInvalidValue;          // refused on the host before this point
    e = launch_embedding(tok, E, h, M, V, D, bf16, st);
    if (e != cudaSuccess) return e;
    NormArgs n2 = na;
    n2.pos = nullptr;
    return launch_rmsnorm(h, g, y, M, D, eps, bf16, st, g_static, &n2);
}

// ------------------------------------------------------------------ RMSNorm / LayerNorm
// y = norm(x) (see the norms above).  One warp per row; lane l owns the float4
// groups l, l+32, ...; kV groups per lane are held in registers (rows up to
// 128*kV floats).
template <int kKind, int kV, bool kBf16>
__global__ void __launch_bounds__(256) k_rmsnorm(const float* __restrict__ x,
                                                 const float* __restrict__ g,
                                                 void* __restrict__ y, int64_t M, int D,
                                                 float eps, NormArgs na) {
    const int lane = threadIdx.x & 31;
    // The gain staged once per CTA for rows of 1024 floats and more (the stores
    // then wait on no global load after the row's reduction): the GQA workload's
    // norms 23.5 -> 18.9 us, the long-context one's 13.0 -> 12.5 us; at 512
    // floats the staging cost more than it saved (8.8 -> 9.5 us), so short rows
    // keep the gain loads.
    constexpr bool kStage = kKind == kNormRms && kBf16 && kV >= 8;
    __shared__ float4 gs[kStage ? kV * 32 : 1];
    pdl_wait();
    pdl_trigger();
    const int n4 = D >> 2;
    if (kStage) {
        for (int c = threadIdx.x; c < n4; c += blockDim.x) gs[c] = __ldg(reinterpret_cast<const float4*>(g) + c);
        __syncthreads();
    }
    const int64_t m = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (m >= M) return;
    const float4* xr = reinterpret_cast<const float4*>(x + m * D);
    float4 v[kV];
#pragma unroll
    for (int i = 0; i < kV; ++i) {
        const int c = lane + 32 * i;
        v[i] = (c < n4) ? xr[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float r = warp_norm_scale<kKind, kV>(v, lane, n4, D, eps);
    const float4* g4 = reinterpret_cast<const float4*>(g);
    const float4* b4 = reinterpret_cast<const float4*>(na.b);
    void* yrow = kBf16 ? (void*)(static_cast<__nv_bfloat16*>(y) + m * D)
                       : (void*)(static_cast<float*>(y) + m * D);
    float* hrow = na.h_out ? na.h_out + m * D : nullptr;
    if (kStage) {
#pragma unroll
        for (int i = 0; i < kV; ++i) {
            const int c = lane + 32 * i;
            if (c >= n4) break;
            const float4 w = gs[c];
            uint2 o;
            o.x = pack_bf16x2(v[i].x * r * w.x, v[i].y * r * w.y);
            o.y = pack_bf16x2(v[i].z * r * w.z, v[i].w * r * w.w);
            reinterpret_cast<uint2*>(yrow)[c] = o;
        }
        return;
    }
#pragma unroll
    for (int i = 0; i < kV; ++i) {
        const int c = lane + 32 * i;
        if (c >= n4) break;
        norm_store<kKind, kBf16>(v[i], r, g4, b4, c, hrow, yrow);
    }
}

// Rows longer than 128*32 floats: passes over the row in global memory (the
// sum for LayerNorm's mean, the sum of squares, the write).
template <bool kBf16>
__global__ void __launch_bounds__(256) k_rmsnorm_long(const float* __restrict__ x,
                                                      const float* __restrict__ g,
                                                      void* __restrict__ y, int64_t M, int D,
                                                      float eps, NormArgs na) {
    const int lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    const int64_t m = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (m >= M) return;
    const float4* xr = reinterpret_cast<const float4*>(x + m * D);
    float mu = 0.f, r = 1.f;
    if (na.kind == kNormLayer) {
        float s = 0.f;
        for (int c = lane; c < D / 4; c += 32) s += sum4(xr[c]);
        mu = warp_sum(s) / (float)D;
    }
    if (na.kind != kNormNone) {
        float ss = 0.f;
        for (int c = lane; c < D / 4; c += 32) {
            float4 t = xr[c];
            t.x -= mu; t.y -= mu; t.z -= mu; t.w -= mu;
            ss += sq4(t);
        }
        r = 1.0f / sqrtf(warp_sum(ss) / (float)D + eps);
    }
    const float4* g4 = reinterpret_cast<const float4*>(g);
    const float4* b4 = reinterpret_cast<const float4*>(na.b);
    void* yrow = kBf16 ? (void*)(static_cast<__nv_bfloat16*>(y) + m * D)
                       : (void*)(static_cast<float*>(y) + m * D);
    float* hrow = na.h_out ? na.h_out + m * D : nullptr;
    for (int c = lane; c < D / 4; c += 32) {
        float4 t = xr[c];
        t.x -= mu; t.y -= mu; t.z -= mu; t.w -= mu;
        if (na.kind == kNormLayer) norm_store<kNormLayer, kBf16>(t, r, g4, b4, c, hrow, yrow);
        else if (na.kind == kNormNone) norm_store<kNormNone, kBf16>(t, r, g4, b4, c, hrow, yrow);
        else norm_store<kNormRms, kBf16>(t, r, g4, b4, c, hrow, yrow);
    }
}

template <int kKind, int kV>
static cudaError_t rms_kind(const float* x, const float* g, void* y, int64_t M, int D, float eps,
                            int out_bf16, const NormArgs& na, cudaStream_t st) {
    const dim3 blocks((unsigned)((M + 7) / 8));
    if (out_bf16)
        return launch_pdl(k_rmsnorm<kKind, kV, true>, blocks, dim3(256), 0, st, x, g, y, M, D, eps,
                          na);
    return launch_pdl(k_rmsnorm<kKind, kV, false>, blocks, dim3(256), 0, st, x, g, y, M, D, eps, na);
}

template <int kV>
static cudaError_t rms_launch(const float* x, const float* g, void* y, int64_t M, int D, float eps,
                              int out_bf16, const NormArgs& na, cudaStream_t st) {
    if (na.kind == kNormLayer) return rms_kind<kNormLayer, kV>(x, g, y, M, D, eps, out_bf16, na, st);
    if (na.kind == kNormNone) return rms_kind<kNormNone, kV>(x, g, y, M, D, eps, out_bf16, na, st);
    return rms_kind<kNormRms, kV>(x, g, y, M, D, eps, out_bf16, na, st);
}

cudaError_t launch_rmsnorm(const float* x, const float* g, void* y, int64_t M, int D, float eps,
                           int out_bf16, cudaStream_t st, int g_static, const NormArgs* nap) {
    if (M <= 0) return cudaSuccess;
    NormArgs na = nap ? *nap : NormArgs{};
    na.pos = nullptr;
    cudaError_t e;
    if (norm_row_launch<false>(&e, nullptr, x, g, nullptr, y, M, 0, D, eps, out_bf16, g_static, na,
                               st))
        return e;
    const int groups = (D / 4 + 31) / 32;   // float4 groups per lane
    if (groups <= 1) return rms_launch<1>(x, g, y, M, D, eps, out_bf16, na, st);
    if (groups <= 2) return rms_launch<2>(x, g, y, M, D, eps, out_bf16, na, st);
    if (groups <= 4) return rms_launch<4>(x, g, y, M, D, eps, out_bf16, na, st);
    if (groups <= 6) return rms_launch<6>(x, g, y, M, D, eps, out_bf16, na, st);
    if (groups <= 8) return rms_launch<8>(x, g, y, M, D, eps, out_bf16, na, st);
    if (groups <= 16) return rms_launch<16>(x, g, y, M, D, eps, out_bf16, na, st);
    if (groups <= 32) return rms_launch<32>(x, g, y, M, D, eps, out_bf16, na, st);
    const dim3 blocks((unsigned)((M + 7) / 8));
    if (out_bf16) return launch_pdl(k_rmsnorm_long<true>, blocks, dim3(256), 0, st, x, g, y, M, D, eps, na);
    return launch_pdl(k_rmsnorm_long<false>, blocks, dim3(256), 0, st, x, g, y, M, D, eps, na);
}

// ------------------------------------------------------------------ RoPE
// In place on x [B, H, S, dh]: the pair (x[2i], x[2i+1]) of token s is turned
// counter-clockwise by pos * theta^(-2i/dh) ("LLM 2", section RoPE: R_i(m)).
// The angle and its sine/cosine are formed in double precision so the result
// does not depend on fp32 angle rounding at large positions.  One thread per pair.
template <typename T>
__global__ void k_rope(T* __restrict__ x, const int32_t* __restrict__ pos, int B, int H, int S,
                       int dh, double log_theta) {
    const int half = dh >> 1;
    const int64_t total = (int64_t)B * H * S * half;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int i = (int)(idx % half);
        const int64_t row = idx / half;                  // (b*H + h)*S + s
        const int s = (int)(row % S);
        const int b = (int)(row / ((int64_t)S * H));
        const double p = pos ? (double)pos[(int64_t)b * S + s] : (double)s;
        const double ang = p * exp(-2.0 * (double)i / (double)dh * log_theta);
        double sd, cd;
        sincos(ang, &sd, &cd);
        const float c = (float)cd, sn = (float)sd;
        T* e = x + row * dh + 2 * i;
        const float x0 = (float)e[0], x1 = (float)e[1];
        const float y0 = x0 * c - x1 * sn, y1 = x0 * sn + x1 * c;
        if constexpr (sizeof(T) == 2) {
            e[0] = __float2bfloat16_rn(y0);
            e[1] = __float2bfloat16_rn(y1);
        } else {
            e[0] = y0;
            e[1] = y1;
        }
    }
}

cudaError_t launch_rope(void* x, const int32_t* pos, int B, int H, int S, int dh, float theta,
                        int is_bf16, cudaStream_t st) {
    const int64_t total = (int64_t)B * H * S * (dh / 2);
    if (total <= 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 32;
    if (blocks > cap) blocks = cap;
    const double lt = log((double)theta);
    if (is_bf16)
        k_rope<__nv_bfloat16><<<(int)blocks, 256, 0, st>>>(static_cast<__nv_bfloat16*>(x), pos, B,
                                                            H, S, dh, lt);
    else
        k_rope<float><<<(int)blocks, 256, 0, st>>>(static_cast<float*>(x), pos, B, H, S, dh, lt);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ self-test
// One warp waits on an mbarrier that expects one arrival nobody makes; the
// bounded wait gives up after limit_ns and latches TFM_ETIMEOUT.
__global__ void k_selftest_wait(uint64_t limit_ns, int* err) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) (void)mbar_wait(b, 0, err, &abort_flag, limit_ns);
    __syncwarp();
}

cudaError_t launch_selftest_wait(uint64_t limit_ns, cudaStream_t st) {
    k_selftest_wait<<<1, 32, 0, st>>>(limit_ns, device_error_word());
    return cudaGetLastError();
}

}  // namespace tfm
