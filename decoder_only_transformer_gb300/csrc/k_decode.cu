// k_decode.cu - attention of one new query per sequence over the KV cache, for
// incremental decoding.
//
// The step after the forward on the generation side ("LLM 2", sections KV cache
// and GQA / MQA): the keys and values of the positions already seen are kept per
// layer, and a new token at position p only computes its own q, k, v; its
// attention is softmax(q k^T / sqrt(dh)) v over positions [0, p] of its kv head
// (CS336 walkthrough, section 5.4, for the last row of the causal mask, where
// nothing is masked).  One query row per (sequence, head) leaves nothing for the
// tensor cores to tile, and the work is reading the cache: the kernel is bound by
// HBM bandwidth, so it runs on the CUDA cores and splits the keys over many CTAs
// (flash-decoding): CTA (b, g, c) takes the G = H / Hkv query heads that read kv
// head g of sequence b against keys [256 c, 256 c + 256), writes the partial row
// max m (log2 domain), row sum l and unnormalised output o per head, and a
// second kernel combines the chunks exactly: with M = max_c m_c,
// o = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c.
#include "common.cuh"
#include "internal.h"

namespace tfm {

namespace {

constexpr int kDecChunk = 256;      // keys per CTA
constexpr int kDecThreads = 128;

template <int DH, int G>
__global__ void __launch_bounds__(kDecThreads) k_decode_partial(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kc,
    const __nv_bfloat16* __restrict__ vc, float* __restrict__ part, int H, int Hkv, int max_seq,
    int L, int nch, float scale_log2) {
    constexpr int NW = kDecThreads / 32;
    __shared__ float qs[G][DH];
    __shared__ float ps[G][kDecChunk];
    __shared__ float red[G][NW];
    __shared__ float osum[NW][G][DH];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = (int)blockIdx.x % nch;
    const int bg = (int)blockIdx.x / nch;            // b * Hkv + g
    const int b = bg / Hkv, g = bg - b * Hkv;
    const int h0 = g * G;                            // first query head of the group
    for (int i = tid; i < G * DH; i += kDecThreads) {
        const int hh = i / DH, d = i - hh * DH;
        qs[hh][d] = __bfloat162float(q[((int64_t)(b * H + h0 + hh)) * DH + d]);
    }
    __syncthreads();
    const int k0 = c * kDecChunk;
    const int n = L - k0 < kDecChunk ? L - k0 : kDecChunk;
    const __nv_bfloat16* kb = kc + ((int64_t)bg * max_seq + k0) * DH;
    const __nv_bfloat16* vb = vc + ((int64_t)bg * max_seq + k0) * DH;

    // Scores: thread t takes keys t, t + 128; each key row is read once for the
    // G heads.
    float mloc[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) mloc[hh] = -INFINITY;
    for (int t = tid; t < kDecChunk; t += kDecThreads) {
        float acc[G];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) acc[hh] = 0.f;
        if (t < n) {
            const uint4* kr = reinterpret_cast<const uint4*>(kb + (int64_t)t * DH);
#pragma unroll
            for (int c8 = 0; c8 < DH / 8; ++c8) {
                const uint4 w = __ldg(kr + c8);
                const float kv[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                                     bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
                for (int hh = 0; hh < G; ++hh)
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[hh] = fmaf(qs[hh][c8 * 8 + e], kv[e], acc[hh]);
            }
        }
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            const float sc = t < n ? acc[hh] * scale_log2 : -INFINITY;
            ps[hh][t] = sc;
            mloc[hh] = fmaxf(mloc[hh], sc);
        }
    }
    // Chunk max per head (n >= 1, so it is finite).
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        float v = mloc[hh];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0) red[hh][warp] = v;
    }
    __syncthreads();
    float mh[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        float v = red[hh][0];
#pragma unroll
        for (int w = 1; w < kDecThreads / 32; ++w) v = fmaxf(v, red[hh][w]);
        mh[hh] = v;
    }
    __syncthreads();
    // p = 2^(s - m) in place and the chunk's row sums.
    float lloc[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) lloc[hh] = 0.f;
    for (int t = tid; t < kDecChunk; t += kDecThreads)
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            const float p = t < n ? exp2f(ps[hh][t] - mh[hh]) : 0.f;
            ps[hh][t] = p;
            lloc[hh] += p;
        }
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        float v = lloc[hh];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[hh][warp] = v;
    }
    __syncthreads();
    // o_h[d] = sum_t p_h[t] v_t[d]: warp w takes keys [64 w, 64 w + 64); lane l
    // reads 16 bytes (8 columns, chunk l % CPR) of rows l / CPR + RPI i, so one
    // warp load covers RPI whole rows and eight loads are in flight per step; a v
    // row is applied to all G heads.  The lanes of a chunk are then summed with
    // shuffles and the four warps through shared memory.
    {
        constexpr int CPR = DH / 8;                  // 16-byte chunks per row
        constexpr int RPI = 32 / CPR;                // rows per warp load
        constexpr int KPW = kDecChunk / NW;          // keys per warp
        const int cl = lane % CPR, rl = lane / CPR;
        float acc[G][8];
#pragma unroll
        for (int hh = 0; hh < G; ++hh)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[hh][e] = 0.f;
        const int t0 = warp * KPW;
        for (int i0 = 0; i0 < KPW; i0 += 8 * RPI) {
            uint4 w[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = t0 + i0 + u * RPI + rl;
                w[u] = t < n ? __ldg(reinterpret_cast<const uint4*>(vb + (int64_t)t * DH) + cl)
                             : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = t0 + i0 + u * RPI + rl;
                const float v8[8] = {bf16_lo(w[u].x), bf16_hi(w[u].x), bf16_lo(w[u].y), bf16_hi(w[u].y),
                                     bf16_lo(w[u].z), bf16_hi(w[u].z), bf16_lo(w[u].w), bf16_hi(w[u].w)};
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const float p = ps[hh][t];           // 0 past n
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[hh][e] = fmaf(p, v8[e], acc[hh][e]);
                }
            }
        }
        // lanes cl, cl + CPR, ... hold the same columns
#pragma unroll
        for (int off = CPR; off < 32; off <<= 1)
#pragma unroll
            for (int hh = 0; hh < G; ++hh)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[hh][e] += __shfl_xor_sync(0xffffffffu, acc[hh][e], off);
        if (rl == 0) {
#pragma unroll
            for (int hh = 0; hh < G; ++hh)
#pragma unroll
                for (int e = 0; e < 8; ++e) osum[warp][hh][cl * 8 + e] = acc[hh][e];
        }
    }
    __syncthreads();
    for (int i = tid; i < G * DH; i += kDecThreads) {
        const int hh = i / DH, d = i - hh * DH;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) v += osum[w][hh][d];
        part[((int64_t)(b * H + h0 + hh) * nch + c) * (DH + 2) + d] = v;
    }
    if (tid < G) {
        float l = 0.f, m = mh[0];
#pragma unroll
        for (int w = 0; w < kDecThreads / 32; ++w) l += red[tid][w];
#pragma unroll
        for (int hh = 1; hh < G; ++hh)
            if (hh == tid) m = mh[hh];                // mh[tid] with constant indices
        float* dst = part + ((int64_t)(b * H + h0 + tid) * nch + c) * (DH + 2);
        dst[DH] = m;
        dst[DH + 1] = l;
    }
}

// One warp per (sequence, head): combine the chunks, write o[b, h*DH + d] bf16.
template <int DH>
__global__ void __launch_bounds__(128) k_decode_combine(const float* __restrict__ part,
                                                       __nv_bfloat16* __restrict__ o, int BH,
                                                       int H, int nch) {
    pdl_wait();
    pdl_trigger();
    const int w = (int)(blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5));
    const int lane = threadIdx.x & 31;
    if (w >= BH) return;
    const float* p = part + (int64_t)w * nch * (DH + 2);
    float M = -INFINITY;
    for (int c = 0; c < nch; ++c) M = fmaxf(M, p[c * (DH + 2) + DH]);
    float acc[DH / 32];
#pragma unroll
    for (int i = 0; i < DH / 32; ++i) acc[i] = 0.f;
    float l = 0.f;
    for (int c = 0; c < nch; ++c) {
        const float* pc = p + c * (DH + 2);
        const float wgt = exp2f(pc[DH] - M);
        l = fmaf(wgt, pc[DH + 1], l);
#pragma unroll
        for (int i = 0; i < DH / 32; ++i) acc[i] = fmaf(wgt, pc[lane + 32 * i], acc[i]);
    }
    const float inv = 1.0f / l;
    const int b = w / H, h = w - b * H;
    __nv_bfloat16* dst = o + (int64_t)b * H * DH + (int64_t)h * DH;
#pragma unroll
    for (int i = 0; i < DH / 32; ++i) dst[lane + 32 * i] = __float2bfloat16_rn(acc[i] * inv);
}

template <int DH, int G>
cudaError_t decode_launch(const void* q, const void* kc, const void* vc, float* part, void* o,
                          int B, int H, int Hkv, int max_seq, int L, float scale,
                          cudaStream_t st) {
    const int nch = (L + kDecChunk - 1) / kDecChunk;
    cudaError_t e = launch_pdl(k_decode_partial<DH, G>, dim3((unsigned)(B * Hkv * nch)),
                               dim3(kDecThreads), 0, st, static_cast<const __nv_bfloat16*>(q),
                               static_cast<const __nv_bfloat16*>(kc),
                               static_cast<const __nv_bfloat16*>(vc), part, H, Hkv, max_seq, L,
                               nch, scale * 1.4426950408889634f);
    if (e != cudaSuccess) return e;
    const int BH = B * H;
    return launch_pdl(k_decode_combine<DH>, dim3((unsigned)((BH + 3) / 4)), dim3(128), 0, st,
                      static_cast<const float*>(part), static_cast<__nv_bfloat16*>(o), BH, H, nch);
}

template <int DH>
cudaError_t decode_dh(const void* q, const void* kc, const void* vc, float* part, void* o, int B,
                      int H, int Hkv, int max_seq, int L, float scale, cudaStream_t st) {
    switch (H / Hkv) {
        case 1: return decode_launch<DH, 1>(q, kc, vc, part, o, B, H, Hkv, max_seq, L, scale, st);
        case 2: return decode_launch<DH, 2>(q, kc, vc, part, o, B, H, Hkv, max_seq, L, scale, st);
        case 4: return decode_launch<DH, 4>(q, kc, vc, part, o, B, H, Hkv, max_seq, L, scale, st);
        case 8: return decode_launch<DH, 8>(q, kc, vc, part, o, B, H, Hkv, max_seq, L, scale, st);
        case 16:
            // 16 heads of 128 columns would need 57.6 KB of static shared memory
            if constexpr (DH <= 64)
                return decode_launch<DH, 16>(q, kc, vc, part, o, B, H, Hkv, max_seq, L, scale, st);
            return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t decode_partial_floats(int B, int H, int max_seq, int dh) {
    return (size_t)B * H * ((max_seq + kDecChunk - 1) / kDecChunk) * (dh + 2);
}

bool decode_supported(int dh, int group) {
    return (dh == 32 || dh == 64 || dh == 128) &&
           (group == 1 || group == 2 || group == 4 || group == 8 || (group == 16 && dh <= 64));
}

cudaError_t launch_decode_attention(const void* q, const void* kc, const void* vc, float* part,
                                    void* o, int B, int H, int Hkv, int max_seq, int L, int dh,
                                    float scale, cudaStream_t st) {
    if (B <= 0 || L <= 0) return cudaSuccess;
    switch (dh) {
        case 32: return decode_dh<32>(q, kc, vc, part, o, B, H, Hkv, max_seq, L, scale, st);
        case 64: return decode_dh<64>(q, kc, vc, part, o, B, H, Hkv, max_seq, L, scale, st);
        case 128: return decode_dh<128>(q, kc, vc, part, o, B, H, Hkv, max_seq, L, scale, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace tfm
