// k_simt.cu - fp32-mode kernels on the CUDA cores (FFMA).  fp32 mode keeps
// every tensor in fp32 so the forward agrees with the fp64 oracle to ~1e-6;
// the tensor cores' tf32 path (10-bit mantissa) could not.  These kernels are
// sized for the small fp32 configurations, not for throughput.
#include "epilogue.cuh"

namespace tfm {

// ------------------------------------------------------------------ GEMM
// C = A[M,K] . B[N,K]^T (bias-free Linear with W stored (out, in), CS336
// walkthrough section 5.3) and, for the SwiGLU epilogue, C2 = A . B2^T in the
// same pass.  64x64 output tile per 256-thread block, k-step 16; thread
// (ty, tx) owns rows 4ty..4ty+3 and the 4 consecutive columns 4tx..4tx+3 (so a
// RoPE pair is always inside one thread).
constexpr int kSimtBM = 64, kSimtBN = 64, kSimtBK = 16;

template <bool kDual>
__global__ void __launch_bounds__(256) k_gemm_simt(const float* __restrict__ A,
                                                   const float* __restrict__ B,
                                                   const float* __restrict__ B2, int M, int N,
                                                   int K, EpiParams epi) {
    __shared__ float As[kSimtBK][kSimtBM + 4];
    __shared__ float Bs[kSimtBK][kSimtBN + 4];
    __shared__ float B2s[kDual ? kSimtBK : 1][kDual ? kSimtBN + 4 : 1];
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int m0 = blockIdx.y * kSimtBM, n0 = blockIdx.x * kSimtBN;
    float acc[4][4] = {}, acc2[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += kSimtBK) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int idx = tid + 256 * i, r = idx >> 4, c = idx & 15;
            const int gk = k0 + c;
            As[c][r] = (m0 + r < M && gk < K) ? A[(int64_t)(m0 + r) * K + gk] : 0.f;
            Bs[c][r] = (n0 + r < N && gk < K) ? B[(int64_t)(n0 + r) * K + gk] : 0.f;
            if (kDual) B2s[c][r] = (n0 + r < N && gk < K) ? B2[(int64_t)(n0 + r) * K + gk] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kSimtBK; ++kk) {
            float a[4], b[4], b2[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = As[kk][ty * 4 + i];
                b[i] = Bs[kk][tx * 4 + i];
                if (kDual) b2[i] = B2s[kk][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
                    if (kDual) acc2[i][j] = fmaf(a[i], b2[j], acc2[i][j]);
                }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) apply_epilogue<4>(epi, m0 + ty * 4 + i, n0 + tx * 4, acc[i], acc2[i]);
}

cudaError_t launch_gemm_simt(const float* A, const float* B, const float* B2, int M, int N, int K,
                             const EpiParams& epi, cudaStream_t st) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    dim3 grid((N + kSimtBN - 1) / kSimtBN, (M + kSimtBM - 1) / kSimtBM);
    if (B2)
        k_gemm_simt<true><<<grid, 256, 0, st>>>(A, B, B2, M, N, K, epi);
    else
        k_gemm_simt<false><<<grid, 256, 0, st>>>(A, B, nullptr, M, N, K, epi);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ attention
// Causal softmax attention in fp32, one warp per (sequence, head, query row).
// Lane l holds coordinates l, l+32, ... of the query and of its output; keys
// 0..i are visited in order with a running max and sum (the stable softmax of
// the CS336 walkthrough section 5.4, evaluated online), so the masked keys
// j > i are never read; with a sliding window w > 0 only keys i-w < j <= i
// ("LLM 2", section 滑动窗口和混合注意力).  o is written with heads merged:
// o[b, i, h*dh + d].
__global__ void __launch_bounds__(256) k_attention_simt(const float* __restrict__ q,
                                                        const float* __restrict__ k,
                                                        const float* __restrict__ v,
                                                        float* __restrict__ o, int B, int H,
                                                        int Hkv, int S, int dh, float scale,
                                                        int window) {
    const int lane = threadIdx.x & 31;
    const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (w >= (int64_t)B * H * S) return;
    const int i = (int)(w % S);
    const int h = (int)((w / S) % H);
    const int b = (int)(w / ((int64_t)S * H));
    const int g = h / (H / Hkv);
    const float* qr = q + (((int64_t)b * H + h) * S + i) * dh;
    const float* kb = k + ((int64_t)b * Hkv + g) * S * dh;
    const float* vb = v + ((int64_t)b * Hkv + g) * S * dh;
    constexpr int kMaxT = 4;                      // dh <= 128
    float qv[kMaxT], acc[kMaxT];
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) {
        const int d = lane + 32 * t;
        qv[t] = d < dh ? qr[d] : 0.f;
        acc[t] = 0.f;
    }
    float mx = -INFINITY, sum = 0.f;
    const int j0 = (window > 0 && i - window + 1 > 0) ? i - window + 1 : 0;
    for (int j = j0; j <= i; ++j) {
        float part = 0.f;
#pragma unroll
        for (int t = 0; t < kMaxT; ++t) {
            const int d = lane + 32 * t;
            if (d < dh) part = fmaf(qv[t], kb[(int64_t)j * dh + d], part);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        const float s = part * scale;
        const float mnew = fmaxf(mx, s);
        const float corr = expf(mx - mnew);       // exp(-inf) = 0 on the first key
        const float p = expf(s - mnew);
        sum = sum * corr + p;
#pragma unroll
        for (int t = 0; t < kMaxT; ++t) {
            const int d = lane + 32 * t;
            if (d < dh) acc[t] = acc[t] * corr + p * vb[(int64_t)j * dh + d];
        }
        mx = mnew;
    }
    float* orow = o + ((int64_t)b * S + i) * ((int64_t)H * dh) + (int64_t)h * dh;
    const float inv = 1.0f / sum;
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) {
        const int d = lane + 32 * t;
        if (d < dh) orow[d] = acc[t] * inv;
    }
}

cudaError_t launch_attention_simt(const float* q, const float* k, const float* v, float* o, int B,
                                  int H, int Hkv, int S, int dh, float scale, cudaStream_t st,
                                  int window) {
    const int64_t warps = (int64_t)B * H * S;
    if (warps <= 0) return cudaSuccess;
    const int64_t blocks = (warps + 7) / 8;
    k_attention_simt<<<(unsigned)blocks, 256, 0, st>>>(q, k, v, o, B, H, Hkv, S, dh, scale, window);
    return cudaGetLastError();
}

}  // namespace tfm
