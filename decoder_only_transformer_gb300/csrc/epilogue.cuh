// epilogue.cuh - what a GEMM does with a chunk of W consecutive accumulator
// columns of one output row.  Shared by the tensor-core GEMM (W = 32, one
// TMEM load per chunk) and the CUDA-core GEMM of fp32 mode (W = 4).
//
// The fusions are the ones the pre-norm block allows without changing what is
// computed:
//  - residual add after the output and down projections (CS336 walkthrough,
//    section 5.7: x = x + attention(norm1(x)); x = x + ffn(norm2(x)));
//  - silu(gate) * up after the W1/W3 projections (section 5.3 SwiGLU);
//  - RoPE on the q and k columns and the head split (B,S,H*dh) -> (B,H,S,dh)
//    after the QKV projection (sections 5.4 多头注意力 and 5.5 RoPE: rotate
//    adjacent pairs of each head by position * theta^(-2i/dh); v is not rotated).
#pragma once

#include "common.cuh"
#include "internal.h"

namespace tfm {

template <int N>
__device__ __forceinline__ void load_vec(const float* p, float (&v)[N]) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            float4 t = *reinterpret_cast<const float4*>(p + i);
            v[i] = t.x; v[i + 1] = t.y; v[i + 2] = t.z; v[i + 3] = t.w;
        }
    } else if constexpr (N % 2 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 2) {
            float2 t = *reinterpret_cast<const float2*>(p + i);
            v[i] = t.x; v[i + 1] = t.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) v[i] = p[i];
    }
}

// Store W values starting at element `col0` of a row (`n_valid` of them are in
// range).  Full chunks use 16-byte (or 8-byte) vector stores.
template <int W>
__device__ __forceinline__ void store_row_f32(float* dst, const float (&v)[W], int n_valid) {
    if (n_valid >= W) {
        if constexpr (W % 4 == 0) {
#pragma unroll
            for (int i = 0; i < W; i += 4)
                *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        } else {
#pragma unroll
            for (int i = 0; i < W; ++i) dst[i] = v[i];
        }
    } else {
#pragma unroll
        for (int i = 0; i < W; ++i)
            if (i < n_valid) dst[i] = v[i];
    }
}

template <int W>
__device__ __forceinline__ void accum_row_f32(float* dst, const float (&v)[W], int n_valid) {
    if (n_valid >= W) {
        if constexpr (W % 4 == 0) {
#pragma unroll
            for (int i = 0; i < W; i += 4) {
                float4 t = *reinterpret_cast<float4*>(dst + i);
                t.x += v[i]; t.y += v[i + 1]; t.z += v[i + 2]; t.w += v[i + 3];
                *reinterpret_cast<float4*>(dst + i) = t;
            }
        } else {
#pragma unroll
            for (int i = 0; i < W; ++i) dst[i] += v[i];
        }
    } else {
#pragma unroll
        for (int i = 0; i < W; ++i)
            if (i < n_valid) dst[i] += v[i];
    }
}

template <int W>
__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const float (&v)[W], int n_valid) {
    if (n_valid >= W) {
        if constexpr (W % 8 == 0) {
#pragma unroll
            for (int i = 0; i < W; i += 8) {
                uint4 t;
                t.x = pack_bf16x2(v[i], v[i + 1]);
                t.y = pack_bf16x2(v[i + 2], v[i + 3]);
                t.z = pack_bf16x2(v[i + 4], v[i + 5]);
                t.w = pack_bf16x2(v[i + 6], v[i + 7]);
                *reinterpret_cast<uint4*>(dst + i) = t;
            }
        } else if constexpr (W % 4 == 0) {
#pragma unroll
            for (int i = 0; i < W; i += 4) {
                uint2 t;
                t.x = pack_bf16x2(v[i], v[i + 1]);
                t.y = pack_bf16x2(v[i + 2], v[i + 3]);
                *reinterpret_cast<uint2*>(dst + i) = t;
            }
        } else {
#pragma unroll
            for (int i = 0; i < W; ++i) dst[i] = __float2bfloat16_rn(v[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < W; ++i)
            if (i < n_valid) dst[i] = __float2bfloat16_rn(v[i]);
    }
}

// Where a QKV column chunk goes: region 0/1/2 = q/k/v, head index, offset in
// the head, and whether it is rotated (q and k are, v is not).
struct QkvSlot {
    int region, head, d0, heads;
};
__device__ __forceinline__ QkvSlot qkv_slot(const EpiParams& p, int col0) {
    const int dh = p.dh, Dq = p.n_head * dh, Dkv = p.n_kv_head * dh;
    QkvSlot r;
    int c = col0;
    if (c >= Dq + Dkv) {
        r.region = 2; c -= Dq + Dkv; r.heads = p.n_kv_head;
    } else if (c >= Dq) {
        r.region = 1; c -= Dq; r.heads = p.n_kv_head;
    } else {
        r.region = 0; r.heads = p.n_head;
    }
    r.head = c / dh;
    r.d0 = c - r.head * dh;
    return r;
}

// Element offset of position s of sequence b in a chunk's head-major buffer: q
// [B, H, S, dh]; k, v the same with n_kv_head heads, or, with kv_stride set, a
// KV cache [B, n_kv_head, kv_stride, dh] at position pos0 + s.
__device__ __forceinline__ int epi_pos0(const EpiParams& p) {
    return p.pos0_dev ? __ldg(p.pos0_dev) : p.pos0;
}
__device__ __forceinline__ int64_t qkv_offset(const EpiParams& p, const QkvSlot& q, int b, int s) {
    const bool cache = q.region > 0 && p.kv_stride > 0;
    const int64_t stride = cache ? p.kv_stride : p.S;
    const int64_t pos = cache ? (int64_t)epi_pos0(p) + s : s;
    return (((int64_t)b * q.heads + q.head) * stride + pos) * p.dh + q.d0;
}

// Output values of one chunk: a = accumulator columns [col0, col0+W) of output
// row `row`; u = the matching "up" columns for EPI_SWIGLU (ignored otherwise).
// For EPI_QKV_ROPE the chunk lies inside one head (W divides dh), col0 % W == 0.
// GELU(z) = z * Phi(z) = 0.5 z (1 + erf(z / sqrt 2)), the exact form ("Chapter 4",
// section 4; CS336 walkthrough (fengye404.top), section 9 GELUFFN).  (A
// five-term erf polynomial, Abramowitz & Stegun 7.1.26, measured no faster in
// the MLP's GEMM epilogue at GPT-2-small widths: 63.9 against 60.8 us.)
__device__ __forceinline__ float gelu_exact(float z) {
    return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f));
}

// kBias = false compiles the bias out (plans without one).
template <int W, bool kBias = true>
__device__ __forceinline__ void epi_compute(const EpiParams& p, int row, int col0,
                                            const float (&a_in)[W], const float (&u)[W],
                                            float (&o)[W]) {
    float a[W];
#pragma unroll
    for (int i = 0; i < W; ++i) a[i] = a_in[i];
    if (kBias && p.bias) {
        if constexpr (W % 4 == 0) {
            if (col0 + W <= p.N) {               // whole chunk: 16-byte loads (bias 16-byte aligned)
                const float4* b4 = reinterpret_cast<const float4*>(p.bias + col0);
#pragma unroll
                for (int i = 0; i < W / 4; ++i) {
                    const float4 t = __ldg(b4 + i);
                    a[4 * i] += t.x; a[4 * i + 1] += t.y; a[4 * i + 2] += t.z; a[4 * i + 3] += t.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < W; ++i)
                    if (col0 + i < p.N) a[i] += __ldg(p.bias + col0 + i);
            }
        } else {
#pragma unroll
            for (int i = 0; i < W; ++i)
                if (col0 + i < p.N) a[i] += __ldg(p.bias + col0 + i);
        }
    }
    if (p.kind == EPI_GELU) {
#pragma unroll
        for (int i = 0; i < W; ++i) o[i] = gelu_exact(a[i]);
    } else if (p.kind == EPI_SWIGLU) {
#pragma unroll
        for (int i = 0; i < W; ++i) o[i] = silu(a[i]) * u[i];
    } else if (p.kind == EPI_QKV_ROPE) {
        const QkvSlot q = qkv_slot(p, col0);
        if (q.region < 2 && row < p.M && p.rope_cs) {
            const int dh = p.dh;
            const int s = epi_pos0(p) + row % p.S;
            float cs[W];                       // (cos, sin) of the W/2 pairs
            load_vec<W>(p.rope_cs + ((int64_t)s * (dh / 2) + q.d0 / 2) * 2, cs);
#pragma unroll
            for (int j = 0; j < W / 2; ++j) {
                const float x0 = a[2 * j], x1 = a[2 * j + 1];
                o[2 * j] = x0 * cs[2 * j] - x1 * cs[2 * j + 1];
                o[2 * j + 1] = x0 * cs[2 * j + 1] + x1 * cs[2 * j];
            }
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j) o[j] = a[j];
        }
    } else {
#pragma unroll
        for (int i = 0; i < W; ++i) o[i] = a[i];
    }
}

// Per-thread global stores of one computed chunk.
template <int W>
__device__ __forceinline__ void epi_store_direct(const EpiParams& p, int row, int col0,
                                                 const float (&o)[W]) {
    if (row >= p.M || col0 >= p.N) return;
    const int n_valid = p.N - col0;
    switch (p.kind) {
        case EPI_STORE_F32:
            store_row_f32<W>(static_cast<float*>(p.out) + (int64_t)row * p.ldo + col0, o, n_valid);
            break;
        case EPI_ACCUM_F32:
            accum_row_f32<W>(static_cast<float*>(p.out) + (int64_t)row * p.ldo + col0, o, n_valid);
            break;
        case EPI_STORE_BF16:
            store_row_bf16<W>(static_cast<__nv_bfloat16*>(p.out) + (int64_t)row * p.ldo + col0, o,
                              n_valid);
            break;
        case EPI_SWIGLU:
        case EPI_GELU:
            if (p.out_bf16)
                store_row_bf16<W>(static_cast<__nv_bfloat16*>(p.out) + (int64_t)row * p.ldo + col0,
                                  o, n_valid);
            else
                store_row_f32<W>(static_cast<float*>(p.out) + (int64_t)row * p.ldo + col0, o,
                                 n_valid);
            break;
        case EPI_QKV_ROPE: {
            const QkvSlot q = qkv_slot(p, col0);
            void* base = q.region == 0 ? p.q : (q.region == 1 ? p.k : p.v);
            const int b = row / p.S, s = row - b * p.S;
            const int64_t off = qkv_offset(p, q, b, s);
            if (p.out_bf16)
                store_row_bf16<W>(static_cast<__nv_bfloat16*>(base) + off, o, W);
            else
                store_row_f32<W>(static_cast<float*>(base) + off, o, W);
            break;
        }
        default:
            break;
    }
}

template <int W>
__device__ __forceinline__ void apply_epilogue(const EpiParams& p, int row, int col0,
                                               const float (&a)[W], const float (&u)[W]) {
    if (row >= p.M || col0 >= p.N) return;
    float o[W];
    epi_compute<W>(p, row, col0, a, u, o);
    epi_store_direct<W>(p, row, col0, o);
}

}  // namespace tfm
