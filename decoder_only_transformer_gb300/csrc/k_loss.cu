// k_loss.cu - the cross-entropy of next-token prediction from per-row
// log-sum-exp statistics, without a pass over materialised logits where the
// LM head's GEMM produced the statistics itself (EPI_LSE).
//
// Per position i with logits z and target t ("LLM 2", section Optimize / Loss;
// CS336 walkthrough (fengye404.top), section 12): lse = log sum_j exp(z_j) and
// loss = lse - z_t, with the maximum taken out before the exponentials.  A row's
// statistics come in slots (max m_k, sum s_k of exp(z - m_k)) over disjoint
// column sets; they merge exactly: M = max_k m_k, sum = sum_k s_k exp(m_k - M),
// lse = M + log(sum).  The mean over all positions is summed by one CTA in a
// fixed order, so it does not depend on timing.
#include "common.cuh"
#include "internal.h"

namespace tfm {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// (m, s) of one set merged into (ma, sa): the result describes both sets.
__device__ __forceinline__ void lse_merge(float& ma, float& sa, float mb, float sb) {
    const float m = fmaxf(ma, mb);
    if (m == -INFINITY) return;                      // both empty
    sa = sa * exp2f((ma - m) * kLog2e) + sb * exp2f((mb - m) * kLog2e);
    ma = m;
}

__device__ __forceinline__ void warp_lse(float& m, float& s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m, o);
        const float so = __shfl_xor_sync(0xffffffffu, s, o);
        lse_merge(m, s, mo, so);
    }
}

// One warp per row of materialised logits: one slot and the target's logit.
__global__ void __launch_bounds__(256) k_lse_rows(const float* __restrict__ logits, int64_t ld,
                                                  int M, int V, const int32_t* __restrict__ targets,
                                                  float2* __restrict__ part,
                                                  float* __restrict__ tgt) {
    pdl_wait();
    pdl_trigger();
    const int row = (int)(blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5));
    const int lane = threadIdx.x & 31;
    if (row >= M) return;
    const float* z = logits + (int64_t)row * ld;
    float m = -INFINITY, s = 0.f;
    for (int j = lane; j < V; j += 32) lse_merge(m, s, z[j], 1.f);
    warp_lse(m, s);
    if (lane == 0) {
        part[row] = make_float2(m, s);
        const int t = targets[row];
        if (t >= 0 && t < V) tgt[row] = z[t];
    }
}

// One warp per row: merge the row's slots, lse and loss.
__global__ void __launch_bounds__(256) k_lse_finish(const float2* __restrict__ part, int slots,
                                                    const float* __restrict__ tgt,
                                                    const int32_t* __restrict__ targets, int M,
                                                    int V, float* __restrict__ loss_out,
                                                    float* __restrict__ lse_out,
                                                    float* __restrict__ loss_tmp, int* err) {
    pdl_wait();
    pdl_trigger();
    const int row = (int)(blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5));
    const int lane = threadIdx.x & 31;
    if (row >= M) return;
    const float2* p = part + (int64_t)row * slots;
    float m = -INFINITY, s = 0.f;
    for (int k = lane; k < slots; k += 32) {
        const float2 v = p[k];
        lse_merge(m, s, v.x, v.y);
    }
    warp_lse(m, s);
    if (lane == 0) {
        const float lse = m + logf(s);
        const int t = targets[row];
        float loss;
        if (t >= 0 && t < V) {
            loss = lse - tgt[row];
        } else {
            loss = __int_as_float(0x7fc00000);       // NaN
            raise_error(err, TFM_EBADTOKEN);
        }
        if (loss_out) loss_out[row] = loss;
        if (lse_out) lse_out[row] = lse;
        loss_tmp[row] = loss;
    }
}

// mean of x[0, M): each thread sums a strided subset in order, then a tree.
__global__ void __launch_bounds__(1024) k_mean(const float* __restrict__ x, int M,
                                               float* __restrict__ out) {
    __shared__ double red[1024];
    pdl_wait();
    pdl_trigger();
    double acc = 0.0;
    for (int i = threadIdx.x; i < M; i += 1024) acc += (double)x[i];
    red[threadIdx.x] = acc;
    __syncthreads();
    for (int w = 512; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) out[0] = (float)(red[0] / (double)M);
}

}  // namespace

cudaError_t launch_lse_rows(const float* logits, int64_t ld, int M, int V, const int32_t* targets,
                            float2* part, float* tgt, cudaStream_t st) {
    if (M <= 0) return cudaSuccess;
    return launch_pdl(k_lse_rows, dim3((unsigned)((M + 7) / 8)), dim3(256), 0, st, logits, ld, M, V,
                      targets, part, tgt);
}

cudaError_t launch_lse_finish(const float2* part, int slots, const float* tgt,
                              const int32_t* targets, int M, int V, float* loss_out,
                              float* lse_out, float* loss_tmp, float* mean_out, cudaStream_t st) {
    if (M <= 0) return cudaSuccess;
    cudaError_t e = launch_pdl(k_lse_finish, dim3((unsigned)((M + 7) / 8)), dim3(256), 0, st, part,
                               slots, tgt, targets, M, V, loss_out, lse_out, loss_tmp,
                               device_error_word());
    if (e != cudaSuccess || !mean_out) return e;
    return launch_pdl(k_mean, dim3(1), dim3(1024), 0, st, static_cast<const float*>(loss_tmp), M,
                      mean_out);
}

}  // namespace tfm
