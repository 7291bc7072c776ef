// k_attention.cu - causal softmax attention for bf16 mode (flash-style).
//
// Computes o = softmax(q k^T / sqrt(dh) + M) v per sequence and head, M = -inf
// above the diagonal (CS336 walkthrough, section 5.4), with query head h
// reading kv head h / (H / Hkv) ("LLM 2", section GQA / MQA).  The softmax is
// evaluated online over key tiles (running row max and sum, rescaling the
// partial output when the max grows), so the S x S score matrix is never
// stored and key tiles entirely above the diagonal are never loaded.  With a
// sliding window w > 0 ("LLM 2", section 滑动窗口和混合注意力: each token sees a
// local band of the causal graph) query i sees keys i-w < j <= i: key tiles
// entirely before the window of the tile's first query are skipped too, and
// the tiles the window edge crosses are masked below it as well.
//
// One CTA = 64 query rows of one (sequence, head); 4 warps x 16 rows.  Key and
// value tiles of 64 rows are double-buffered in shared memory with cp.async
// (zero-filled past the sequence end).  Both products run on the tensor cores
// with mma.sync m16n8k16 (bf16 in, fp32 accumulate); the score fragments are
// reused in registers as the A operand of P.V.  Heavy (late) query tiles of
// every head are scheduled before any light one.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace tfm {

namespace {

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// D (16x8 fp32) += A (16x16 bf16, row) . B (16x8 bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

constexpr int kAttBM = 64;   // query rows per CTA
constexpr int kAttBN = 64;   // keys per tile

template <int DH>
struct AttSmem {
    static constexpr int kLd = DH + 8;                       // padded row, in elements
    static constexpr int kTile = kAttBN * kLd;               // elements per K or V tile
    static constexpr int kBytes = (kAttBM * kLd + 4 * kTile) * 2;
};

template <int DH>
__global__ void __launch_bounds__(128) k_attention_mma(const __nv_bfloat16* __restrict__ q,
                                                       const __nv_bfloat16* __restrict__ k,
                                                       const __nv_bfloat16* __restrict__ v,
                                                       __nv_bfloat16* __restrict__ o, int H,
                                                       int Hkv, int S, float scale_log2,
                                                       int window) {
    using L = AttSmem<DH>;
    constexpr int LD = L::kLd;
    extern __shared__ __align__(16) __nv_bfloat16 att_smem[];
    __nv_bfloat16* Qs = att_smem;
    __nv_bfloat16* Ks = att_smem + kAttBM * LD;            // [2][BN][LD]
    __nv_bfloat16* Vs = Ks + 2 * L::kTile;                  // [2][BN][LD]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_wait();
    pdl_trigger();
    const int num_qt = (S + kAttBM - 1) / kAttBM;
    // 1-D grid ordered heaviest first across all (sequence, head) (longest first).
    const int BH = (int)gridDim.x / num_qt;
    const int qt = num_qt - 1 - (int)blockIdx.x / BH;
    const int bh = (int)blockIdx.x % BH, b = bh / H, h = bh - b * H;
    const int g = h / (H / Hkv);
    const __nv_bfloat16* qg = q + ((int64_t)(b * H + h) * S) * DH;
    const __nv_bfloat16* kg = k + ((int64_t)(b * Hkv + g) * S) * DH;
    const __nv_bfloat16* vg = v + ((int64_t)(b * Hkv + g) * S) * DH;

    auto load_tile = [&](__nv_bfloat16* dst, const __nv_bfloat16* src, int r0) {
        constexpr int CH = DH / 8;                          // 16-byte chunks per row
        for (int i = tid; i < kAttBN * CH; i += 128) {
            const int r = i / CH, c = i - r * CH;
            const int gr = r0 + r;
            const __nv_bfloat16* sp = src + (int64_t)(gr < S ? gr : S - 1) * DH + c * 8;
            cp_async16(smem_u32(dst + r * LD + c * 8), sp, gr < S ? 16u : 0u);
        }
    };

    // First key tile: the one holding the window start of the tile's first query.
    const int q0 = qt * kAttBM;
    const int jbeg = (window > 0 && q0 - window + 1 > 0) ? (q0 - window + 1) / kAttBN : 0;
    // Tiles below this key index can hold keys before some row's window start.
    const int win_lo = window > 0 ? q0 + kAttBM - window : INT_MIN;
    load_tile(Qs, qg, q0);
    cp_async_commit();
    load_tile(Ks + (jbeg & 1) * L::kTile, kg, jbeg * kAttBN);
    load_tile(Vs + (jbeg & 1) * L::kTile, vg, jbeg * kAttBN);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    // Query fragments of this warp's 16 rows, all of dh, kept in registers.
    uint32_t qf[DH / 16][4];
#pragma unroll
    for (int kc = 0; kc < DH / 16; ++kc)
        ldsm_x4(smem_u32(Qs + (warp * 16 + (lane & 15)) * LD + kc * 16 + (lane >> 4) * 8), qf[kc]);

    float oacc[DH / 8][4];
#pragma unroll
    for (int i = 0; i < DH / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY;              // running max (log2 domain), rows g, g+8
    float l_lo = 0.f, l_hi = 0.f;                           // this thread's partial row sums
    const int row_lo = qt * kAttBM + warp * 16 + (lane >> 2);
    const int row_hi = row_lo + 8;

    for (int j = jbeg; j <= qt; ++j) {
        const int buf = j & 1;
        if (j + 1 <= qt) {
            load_tile(Ks + (buf ^ 1) * L::kTile, kg, (j + 1) * kAttBN);
            load_tile(Vs + (buf ^ 1) * L::kTile, vg, (j + 1) * kAttBN);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const __nv_bfloat16* Kt = Ks + buf * L::kTile;
        const __nv_bfloat16* Vt = Vs + buf * L::kTile;

        // S = Q K^T for 16 rows x 64 keys (8 blocks of 8 keys).
        float s[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
        for (int kc = 0; kc < DH / 16; ++kc) {
#pragma unroll
            for (int nb2 = 0; nb2 < 4; ++nb2) {
                uint32_t r[4];
                ldsm_x4(smem_u32(Kt + (nb2 * 16 + (lane >> 4) * 8 + (lane & 7)) * LD + kc * 16 +
                                 ((lane >> 3) & 1) * 8),
                        r);
                mma_bf16_16816(s[2 * nb2], qf[kc], r[0], r[1]);
                mma_bf16_16816(s[2 * nb2 + 1], qf[kc], r[2], r[3]);
            }
        }

        // Mask keys above the diagonal and past S: only the diagonal tile and a
        // tile reaching past S need it (warp-uniform test).
        if (j == qt || (j + 1) * kAttBN > S) {
            const int key0 = j * kAttBN + 2 * (lane & 3);
#pragma unroll
            for (int nb = 0; nb < 8; ++nb)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = key0 + nb * 8 + e;
                    if (key > row_lo || key >= S) s[nb][e] = -INFINITY;
                    if (key > row_hi || key >= S) s[nb][2 + e] = -INFINITY;
                }
        }
        // Keys before a row's window (a row left with none in this tile keeps
        // the -inf max, handled below as for the causal mask).
        if (j * kAttBN < win_lo) {
            const int key0 = j * kAttBN + 2 * (lane & 3);
#pragma unroll
            for (int nb = 0; nb < 8; ++nb)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = key0 + nb * 8 + e;
                    if (key <= row_lo - window) s[nb][e] = -INFINITY;
                    if (key <= row_hi - window) s[nb][2 + e] = -INFINITY;
                }
        }
        // Row max of the raw scores (the scale is positive, so it commutes with
        // the max), three-input maxima, then across the four lanes of a row.
        float mx_lo = fmaxf(s[0][0], s[0][1]), mx_hi = fmaxf(s[0][2], s[0][3]);
#pragma unroll
        for (int nb = 1; nb < 8; ++nb) {
            mx_lo = fmax3(mx_lo, s[nb][0], s[nb][1]);
            mx_hi = fmax3(mx_hi, s[nb][2], s[nb][3]);
        }
        mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
        mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
        mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
        mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
        mx_lo = fmaxf(m_lo, mx_lo * scale_log2);
        mx_hi = fmaxf(m_hi, mx_hi * scale_log2);
        const float base_lo = (mx_lo == -INFINITY) ? 0.f : mx_lo;
        const float base_hi = (mx_hi == -INFINITY) ? 0.f : mx_hi;
        const float corr_lo = fast_exp2(m_lo - base_lo), corr_hi = fast_exp2(m_hi - base_hi);
        m_lo = mx_lo;
        m_hi = mx_hi;
        l_lo *= corr_lo;
        l_hi *= corr_hi;
#pragma unroll
        for (int i = 0; i < DH / 8; ++i) {
            oacc[i][0] *= corr_lo; oacc[i][1] *= corr_lo;
            oacc[i][2] *= corr_hi; oacc[i][3] *= corr_hi;
        }
        // p = 2^(s*scale - base): one FMA and one exponential per score.
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
            s[nb][0] = fast_exp2(fmaf(s[nb][0], scale_log2, -base_lo));
            s[nb][1] = fast_exp2(fmaf(s[nb][1], scale_log2, -base_lo));
            s[nb][2] = fast_exp2(fmaf(s[nb][2], scale_log2, -base_hi));
            s[nb][3] = fast_exp2(fmaf(s[nb][3], scale_log2, -base_hi));
            l_lo += s[nb][0] + s[nb][1];
            l_hi += s[nb][2] + s[nb][3];
        }

        // O += P V: P (bf16) straight from the score fragments.
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            uint32_t a[4];
            a[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
            a[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
            a[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            a[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
            for (int db2 = 0; db2 < DH / 16; ++db2) {
                uint32_t r[4];
                ldsm_x4_t(smem_u32(Vt + (kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7)) * LD +
                                   db2 * 16 + (lane >> 4) * 8),
                          r);
                mma_bf16_16816(oacc[2 * db2], a, r[0], r[1]);
                mma_bf16_16816(oacc[2 * db2 + 1], a, r[2], r[3]);
            }
        }
        __syncthreads();
    }

    // Normalise and write o[b, s, h*dh + d] (heads merged back).
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
    const float inv_lo = 1.0f / l_lo, inv_hi = 1.0f / l_hi;
    const int64_t ld_o = (int64_t)H * DH;
    const int d0 = 2 * (lane & 3);
#pragma unroll
    for (int db = 0; db < DH / 8; ++db) {
        const int d = h * DH + db * 8 + d0;
        if (row_lo < S)
            *reinterpret_cast<uint32_t*>(o + ((int64_t)b * S + row_lo) * ld_o + d) =
                pack_bf16x2(oacc[db][0] * inv_lo, oacc[db][1] * inv_lo);
        if (row_hi < S)
            *reinterpret_cast<uint32_t*>(o + ((int64_t)b * S + row_hi) * ld_o + d) =
                pack_bf16x2(oacc[db][2] * inv_hi, oacc[db][3] * inv_hi);
    }
}

template <int DH>
cudaError_t launch_dh(const void* q, const void* k, const void* v, void* o, int B, int H, int Hkv,
                      int S, float scale, int window, cudaStream_t st) {
    using L = AttSmem<DH>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_attention_mma<DH>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dim3 grid(((S + kAttBM - 1) / kAttBM) * B * H);
    return launch_pdl(k_attention_mma<DH>, grid, dim3(128), L::kBytes, st,
                      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
                      static_cast<const __nv_bfloat16*>(v), static_cast<__nv_bfloat16*>(o), H, Hkv,
                      S, scale * 1.4426950408889634f, window);
}

}  // namespace

cudaError_t launch_attention_bf16(const void* q, const void* k, const void* v, void* o, int B,
                                  int H, int Hkv, int S, int dh, float scale, cudaStream_t st,
                                  int window) {
    if (B <= 0 || S <= 0) return cudaSuccess;
    if (window >= S) window = 0;                        // the whole prefix: plain causal
    switch (dh) {
        case 32: return launch_dh<32>(q, k, v, o, B, H, Hkv, S, scale, window, st);
        case 64: return launch_dh<64>(q, k, v, o, B, H, Hkv, S, scale, window, st);
        case 128: return launch_dh<128>(q, k, v, o, B, H, Hkv, S, scale, window, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace tfm
