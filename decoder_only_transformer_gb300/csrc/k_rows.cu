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

// ------------------------------------------------------------------ embedding + RMSNorm
// The forward's first two steps in one pass: h[m] = E[tok[m]] (fp32 residual
// stream) and y[m] = h[m] / sqrt(mean(h[m]^2) + eps) * g (the first block's
// input norm), the row held in registers in between.  One warp per row; lane l
// owns the 4-float groups l, l+32, ...; an id outside [0, V) writes zeros and
// raises TFM_EBADTOKEN.
template <int kV, bool kBf16E, bool kBf16Y>
__global__ void __launch_bounds__(256) k_embed_rmsnorm(const int32_t* __restrict__ tok,
                                                       const void* __restrict__ E,
                                                       const float* __restrict__ g,
                                                       float* __restrict__ h, void* __restrict__ y,
                                                       int64_t M, int V, int D, float eps,
                                                       int* err) {
    const int lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    const int64_t m = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (m >= M) return;
    const int n4 = D >> 2;
    const int t = __ldg(tok + m);
    const bool ok = (t >= 0 && t < V);
    if (!ok && lane == 0) raise_error(err, TFM_EBADTOKEN);
    const int64_t row = ok ? t : 0;
    float4 v[kV];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kV; ++i) {
        const int c = lane + 32 * i;
        v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < n4 && ok) {
            if (kBf16E) {
                const uint2 w = __ldg(reinterpret_cast<const uint2*>(
                                          static_cast<const __nv_bfloat16*>(E) + row * D) + c);
                v[i] = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
            } else {
                v[i] = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(E) + row * D) + c);
            }
        }
        if (c < n4) reinterpret_cast<float4*>(h + m * D)[c] = v[i];
        ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = 1.0f / sqrtf(ss / (float)D + eps);
    const float4* g4 = reinterpret_cast<const float4*>(g);
#pragma unroll
    for (int i = 0; i < kV; ++i) {
        const int c = lane + 32 * i;
        if (c >= n4) break;
        const float4 w = __ldg(g4 + c);
        const float a0 = v[i].x * r * w.x, a1 = v[i].y * r * w.y;
        const float a2 = v[i].z * r * w.z, a3 = v[i].w * r * w.w;
        if (kBf16Y) {
            uint2 o;
            o.x = pack_bf16x2(a0, a1);
            o.y = pack_bf16x2(a2, a3);
            reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(y) + m * D)[c] = o;
        } else {
            reinterpret_cast<float4*>(static_cast<float*>(y) + m * D)[c] = make_float4(a0, a1, a2, a3);
        }
    }
}

// ------------------------------------------------------------------ few rows
// For a handful of rows (a decode step has one per sequence) the warp-per-row
// kernels leave the latency of each dependent load exposed.  Here one CTA of 256
// threads takes a row: thread t owns the 4-float groups t, t + 256, ... (kPer of
// them); a model's gain is a weight that no launch writes, so it is loaded
// before the dependency wait (g_static); the sum of squares is reduced over the
// block.
// kEmbed: the row is E[tok[m]] (fp32 or bf16), also written to h, as in
// k_embed_rmsnorm.
constexpr int kRowKernelMaxM = 64;

template <int kPer, bool kEmbed, bool kBf16E, bool kBf16Y>
__global__ void __launch_bounds__(256) k_norm_row(const int32_t* __restrict__ tok,
                                                  const void* __restrict__ X,
                                                  const float* __restrict__ g,
                                                  float* __restrict__ h, void* __restrict__ y,
                                                  int V, int D, float eps, int g_static,
                                                  int* err) {
    __shared__ float red[8];
    const int tid = threadIdx.x, lane = tid & 31;
    const int64_t m = blockIdx.x;
    const int n4 = D >> 2;
    const float4* g4 = reinterpret_cast<const float4*>(g);
    float4 gv[kPer];
    if (!g_static) pdl_wait();                   // g may come from the launch before
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int c = tid + 256 * i;
        gv[i] = c < n4 ? __ldg(g4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
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
    float4 v[kPer];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int c = tid + 256 * i;
        v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < n4 && ok) {
            if (kBf16E) {
                const uint2 w = __ldg(reinterpret_cast<const uint2*>(
                                          static_cast<const __nv_bfloat16*>(X) + row * D) + c);
                v[i] = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
            } else {
                v[i] = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(X) + row * D) + c);
            }
        }
        if (kEmbed && c < n4) reinterpret_cast<float4*>(h + m * D)[c] = v[i];
        ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[tid >> 5] = ss;
    __syncthreads();
    ss = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) ss += red[w];
    const float r = 1.0f / sqrtf(ss / (float)D + eps);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int c = tid + 256 * i;
        if (c >= n4) continue;
        const float4 w = gv[i];
        const float a0 = v[i].x * r * w.x, a1 = v[i].y * r * w.y;
        const float a2 = v[i].z * r * w.z, a3 = v[i].w * r * w.w;
        if (kBf16Y) {
            uint2 o;
            o.x = pack_bf16x2(a0, a1);
            o.y = pack_bf16x2(a2, a3);
            reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(y) + m * D)[c] = o;
        } else {
            reinterpret_cast<float4*>(static_cast<float*>(y) + m * D)[c] = make_float4(a0, a1, a2, a3);
        }
    }
}

// Few-row launch (M <= kRowKernelMaxM, D <= 8192); returns false when it does not apply.
template <bool kEmbed>
static bool norm_row_launch(cudaError_t* e, const int32_t* tok, const void* X, const float* g,
                            float* h, void* y, int64_t M, int V, int D, float eps, int bf16,
                            int g_static, cudaStream_t st) {
    if (M > kRowKernelMaxM || D > 8192) return false;
    const int per = (D / 4 + 255) / 256;
    const dim3 grid((unsigned)M), block(256);
    int* err = device_error_word();
#define TFM_ROW_LAUNCH(P)                                                                        \
    *e = bf16 ? launch_pdl(k_norm_row<P, kEmbed, kEmbed, true>, grid, block, 0, st, tok, X, g, h, \
                           y, V, D, eps, g_static, err)                                           \
              : launch_pdl(k_norm_row<P, kEmbed, false, false>, grid, block, 0, st, tok, X, g, h, \
                           y, V, D, eps, g_static, err)
    if (per <= 1) TFM_ROW_LAUNCH(1);
    else if (per <= 2) TFM_ROW_LAUNCH(2);
    else if (per <= 4) TFM_ROW_LAUNCH(4);
    else TFM_ROW_LAUNCH(8);
#undef TFM_ROW_LAUNCH
    return true;
}

template <int kV>
cudaError_t embed_norm_launch(const int32_t* tok, const void* E, const float* g, float* h, void* y,
                              int64_t M, int V, int D, float eps, int bf16, cudaStream_t st) {
    const dim3 blocks((unsigned)((M + 7) / 8));
    if (bf16)
        return launch_pdl(k_embed_rmsnorm<kV, true, true>, blocks, dim3(256), 0, st, tok, E, g, h,
                          y, M, V, D, eps, device_error_word());
    return launch_pdl(k_embed_rmsnorm<kV, false, false>, blocks, dim3(256), 0, st, tok, E, g, h, y,
                      M, V, D, eps, device_error_word());
}

cudaError_t launch_embed_rmsnorm(const int32_t* tok, const void* E, const float* g, float* h,
                                 void* y, int64_t M, int V, int D, float eps, int bf16,
                                 cudaStream_t st, int g_static) {
    if (M <= 0) return cudaSuccess;
    cudaError_t e;
    if (norm_row_launch<true>(&e, tok, E, g, h, y, M, V, D, eps, bf16, g_static, st)) return e;
    const int groups = (D / 4 + 31) / 32;   // 4-float groups per lane
    if (groups <= 1) return embed_norm_launch<1>(tok, E, g, h, y, M, V, D, eps, bf16, st);
    if (groups <= 2) return embed_norm_launch<2>(tok, E, g, h, y, M, V, D, eps, bf16, st);
    if (groups <= 4) return embed_norm_launch<4>(tok, E, g, h, y, M, V, D, eps, bf16, st);
    if (groups <= 8) return embed_norm_launch<8>(tok, E, g, h, y, M, V, D, eps, bf16, st);
    if (groups <= 16) return embed_norm_launch<16>(tok, E, g, h, y, M, V, D, eps, bf16, st);
    if (groups <= 32) return embed_norm_launch<32>(tok, E, g, h, y, M, V, D, eps, bf16, st);
    // Rows beyond 4096: the gather and the norm as two launches.
    e = launch_embedding(tok, E, h, M, V, D, bf16, st);
    if (e != cudaSuccess) return e;
    return launch_rmsnorm(h, g, y, M, D, eps, bf16, st);
}

// ------------------------------------------------------------------ RMSNorm
// y = x / sqrt(mean(x^2) + eps) * g, in fp32, rounded once to the output type
// (CS336 walkthrough, section 5.6: fp32 through the gain multiply, then cast).
// One warp per row; lane l owns the float4 groups l, l+32, ...; kV groups per
// lane are held in registers (rows up to 128*kV floats).
template <int kV, bool kBf16>
__global__ void __launch_bounds__(256) k_rmsnorm(const float* __restrict__ x,
                                                 const float* __restrict__ g,
                                                 void* __restrict__ y, int64_t M, int D,
                                                 float eps) {
    const int lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    const int64_t m = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (m >= M) return;
    const int n4 = D >> 2;
    const float4* xr = reinterpret_cast<const float4*>(x + m * D);
    float4 v[kV];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kV; ++i) {
        const int c = lane + 32 * i;
        v[i] = (c < n4) ? xr[c] : make_float4(0.f, 0.f, 0.f, 0.f);
        ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = 1.0f / sqrtf(ss / (float)D + eps);
    const float4* g4 = reinterpret_cast<const float4*>(g);
#pragma unroll
    for (int i = 0; i < kV; ++i) {
        const int c = lane + 32 * i;
        if (c >= n4) break;
        const float4 w = __ldg(g4 + c);
        const float a0 = v[i].x * r * w.x, a1 = v[i].y * r * w.y;
        const float a2 = v[i].z * r * w.z, a3 = v[i].w * r * w.w;
        if (kBf16) {
            uint2 o;
            o.x = pack_bf16x2(a0, a1);
            o.y = pack_bf16x2(a2, a3);
            reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(y) + m * D)[c] = o;
        } else {
            reinterpret_cast<float4*>(static_cast<float*>(y) + m * D)[c] = make_float4(a0, a1, a2, a3);
        }
    }
}

// Rows longer than 128*32 floats: two passes over the row.
template <bool kBf16>
__global__ void __launch_bounds__(256) k_rmsnorm_long(const float* __restrict__ x,
                                                      const float* __restrict__ g,
                                                      void* __restrict__ y, int64_t M, int D,
                                                      float eps) {
    const int lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    const int64_t m = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (m >= M) return;
    const float4* xr = reinterpret_cast<const float4*>(x + m * D);
    float ss = 0.f;
    for (int c = lane; c < D / 4; c += 32) {
        const float4 t = xr[c];
        ss += t.x * t.x + t.y * t.y + t.z * t.z + t.w * t.w;
    }
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = 1.0f / sqrtf(ss / (float)D + eps);
    for (int c = lane; c < D / 4; c += 32) {
        const float4 t = xr[c], w = reinterpret_cast<const float4*>(g)[c];
        const float a0 = t.x * r * w.x, a1 = t.y * r * w.y, a2 = t.z * r * w.z, a3 = t.w * r * w.w;
        if (kBf16) {
            uint2 o;
            o.x = pack_bf16x2(a0, a1);
            o.y = pack_bf16x2(a2, a3);
            reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(y) + m * D)[c] = o;
        } else {
            reinterpret_cast<float4*>(static_cast<float*>(y) + m * D)[c] = make_float4(a0, a1, a2, a3);
        }
    }
}

template <int kV>
static cudaError_t rms_launch(const float* x, const float* g, void* y, int64_t M, int D, float eps,
                              int out_bf16, cudaStream_t st) {
    const dim3 blocks((unsigned)((M + 7) / 8));
    if (out_bf16) return launch_pdl(k_rmsnorm<kV, true>, blocks, dim3(256), 0, st, x, g, y, M, D, eps);
    return launch_pdl(k_rmsnorm<kV, false>, blocks, dim3(256), 0, st, x, g, y, M, D, eps);
}

cudaError_t launch_rmsnorm(const float* x, const float* g, void* y, int64_t M, int D, float eps,
                           int out_bf16, cudaStream_t st, int g_static) {
    if (M <= 0) return cudaSuccess;
    cudaError_t e;
    if (norm_row_launch<false>(&e, nullptr, x, g, nullptr, y, M, 0, D, eps, out_bf16, g_static, st))
        return e;
    const int groups = (D / 4 + 31) / 32;   // float4 groups per lane
    if (groups <= 1) return rms_launch<1>(x, g, y, M, D, eps, out_bf16, st);
    if (groups <= 2) return rms_launch<2>(x, g, y, M, D, eps, out_bf16, st);
    if (groups <= 4) return rms_launch<4>(x, g, y, M, D, eps, out_bf16, st);
    if (groups <= 6) return rms_launch<6>(x, g, y, M, D, eps, out_bf16, st);
    if (groups <= 8) return rms_launch<8>(x, g, y, M, D, eps, out_bf16, st);
    if (groups <= 16) return rms_launch<16>(x, g, y, M, D, eps, out_bf16, st);
    if (groups <= 32) return rms_launch<32>(x, g, y, M, D, eps, out_bf16, st);
    const dim3 blocks((unsigned)((M + 7) / 8));
    if (out_bf16) return launch_pdl(k_rmsnorm_long<true>, blocks, dim3(256), 0, st, x, g, y, M, D, eps);
    return launch_pdl(k_rmsnorm_long<false>, blocks, dim3(256), 0, st, x, g, y, M, D, eps);
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
