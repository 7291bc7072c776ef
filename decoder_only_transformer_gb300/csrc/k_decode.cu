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
// head g of sequence b against the c-th chunk of NK = 8192 / dh keys, writes the
// partial row max m (log2 domain), row sum l and unnormalised output o per head,
// and a second kernel combines the chunks exactly: with M = max_c m_c,
// o = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c.
//
// Bandwidth comes from bytes in flight: a CTA fetches its whole K and V chunk
// (16 KB each, contiguous in the cache layout) with two bulk asynchronous copies
// at its start, so the chunk costs one DRAM round trip instead of one per load
// wave, and several CTAs per SM keep ~150 KB per SM in flight.  (Chunks of 32 KB
// measured slower at long caches: long 176.9 vs 182.0 us per step, gpt2s 426.4 vs
// 433.6 us; 8 KB slower again at gqa, whose 17 MB per layer are over 256 CTAs
// either way.)  Positions before
// the new one were written by earlier launches and are copied before the grid
// dependency wait, overlapping the QKV projection's tail; the new token's row
// (written by the launch just before) and q are read after it.  The math then
// reads shared memory with DH/8 lanes per key row (16 bytes each: one row per
// group of lanes, conflict-free), reducing the dot products with shuffles.
#include "common.cuh"
#include "internal.h"

namespace tfm {

namespace {

constexpr int kDecThreads = 128;
constexpr int kDecNW = kDecThreads / 32;
__host__ __device__ constexpr int dec_keys(int dh) { return 8192 / dh; }   // keys per CTA: 16 KB of K

// Dynamic shared memory of one CTA.
template <int DH, int G>
struct DecSmem {
    static constexpr int kKeys = dec_keys(DH);
    static constexpr int kK = 0;                              // bf16 [kKeys][DH]
    static constexpr int kV = kKeys * DH * 2;                 // bf16 [kKeys][DH]
    static constexpr int kP = 2 * kKeys * DH * 2;             // fp32 [G][kKeys] scores, then p
    static constexpr int kO = kP + G * kKeys * 4;             // fp32 [NW][G][DH] per-warp o
    static constexpr int kRedM = kO + kDecNW * G * DH * 4;    // fp32 [G][NW]
    static constexpr int kRedL = kRedM + G * kDecNW * 4;      // fp32 [G][NW]
    static constexpr int kBar = kRedL + G * kDecNW * 4;       // mbarrier
    static constexpr int kBytes = kBar + 16;
};

template <int DH, int G>
__global__ void __launch_bounds__(kDecThreads) k_decode_partial(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kc,
    const __nv_bfloat16* __restrict__ vc, float* __restrict__ part, __nv_bfloat16* __restrict__ o,
    int H, int Hkv, int max_seq, const int* __restrict__ pos_dev, int nch, float scale_log2,
    int window, int* err) {
    using Sm = DecSmem<DH, G>;
    constexpr int NK = Sm::kKeys, NW = kDecNW;
    constexpr int CPR = DH / 8;                      // lanes per key row, 16 bytes each
    constexpr int RPW = 32 / CPR;                    // rows per warp step
    constexpr int STEPS = NK / (NW * RPW);
    extern __shared__ __align__(128) uint8_t sm[];
    __shared__ int abort_flag;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar = sbase + Sm::kBar;
    float* ps = reinterpret_cast<float*>(sm + Sm::kP);
    float* osum = reinterpret_cast<float*>(sm + Sm::kO);
    float* red_m = reinterpret_cast<float*>(sm + Sm::kRedM);
    float* red_l = reinterpret_cast<float*>(sm + Sm::kRedL);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cl = lane % CPR, rl = lane / CPR;
    const int c = (int)blockIdx.x % nch;
    const int bg = (int)blockIdx.x / nch;            // b * Hkv + g
    // The position pos of the new token was stored before the launches of this
    // step's earlier layers, and the cache rows [0, pos) by earlier steps (or the
    // prefill), all complete before the launch before this one could start.
    const int pos = __ldg(pos_dev);
    const int k0 = c * NK;
    // attended keys [ws, pos]: ws = 0, or the sliding window's first key
    const int ws = (window > 0 && pos - window + 1 > 0) ? pos - window + 1 : 0;
    if (k0 > pos || k0 + NK <= ws) return;           // chunk outside the attended keys
    const int n = min(NK, pos + 1 - k0);             // keys of this chunk
    const int nprev = min(NK, pos - k0);             // of them, those cached before this step
    const int b = bg / Hkv, g = bg - b * Hkv;
    const int h0 = g * G;                            // first query head of the group
    const __nv_bfloat16* kb = kc + ((int64_t)bg * max_seq + k0) * DH;
    const __nv_bfloat16* vb = vc + ((int64_t)bg * max_seq + k0) * DH;
    if (tid == 0) {
        abort_flag = 0;
        mbar_init(bar, 1);
        fence_mbar_init();
        if (nprev > 0) {
            const uint32_t bytes = (uint32_t)nprev * DH * 2;
            mbar_arrive_expect_tx(bar, 2 * bytes);
            bulk_load(sbase + Sm::kK, kb, bytes, bar);
            bulk_load(sbase + Sm::kV, vb, bytes, bar);
        } else {
            mbar_arrive(bar);
        }
    }
    pdl_wait();
    pdl_trigger();
    // The new token's k, v row and q, written by the QKV projection just before.
    if (pos - k0 < NK && tid < 2 * CPR) {
        const int r = pos - k0, part_ = tid / CPR, ch = tid % CPR;
        const uint4 w = __ldg(reinterpret_cast<const uint4*>((part_ ? vb : kb) + (int64_t)r * DH) + ch);
        *reinterpret_cast<uint4*>(sm + (part_ ? Sm::kV : Sm::kK) + r * DH * 2 + ch * 16) = w;
    }
    float qv[G][8];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(q + ((int64_t)(b * H + h0 + hh)) * DH) + cl);
        qv[hh][0] = bf16_lo(w.x); qv[hh][1] = bf16_hi(w.x);
        qv[hh][2] = bf16_lo(w.y); qv[hh][3] = bf16_hi(w.y);
        qv[hh][4] = bf16_lo(w.z); qv[hh][5] = bf16_hi(w.z);
        qv[hh][6] = bf16_lo(w.w); qv[hh][7] = bf16_hi(w.w);
    }
    __syncthreads();                                  // barrier initialised, new row stored
    const bool ok = mbar_wait(bar, 0, err, &abort_flag);
    if (!__syncthreads_and(ok)) return;              // timed out: the error word is set

    // Scores s_h(t) = q_h . k_t (log2 domain): a row per group of CPR lanes.
    float mloc[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) mloc[hh] = -INFINITY;
#pragma unroll 4
    for (int st = 0; st < STEPS; ++st) {
        const int row = (st * NW + warp) * RPW + rl;
        const uint4 w = *reinterpret_cast<const uint4*>(sm + Sm::kK + row * DH * 2 + cl * 16);
        const float kv[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                             bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
        float d[G];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            float a = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) a = fmaf(qv[hh][e], kv[e], a);
            d[hh] = a;
        }
#pragma unroll
        for (int off = 1; off < CPR; off <<= 1)
#pragma unroll
            for (int hh = 0; hh < G; ++hh) d[hh] += __shfl_xor_sync(0xffffffffu, d[hh], off);
        if (cl == 0) {
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                // rows >= n unused; rows before the window start masked
                const float sc = (row < n && k0 + row >= ws) ? d[hh] * scale_log2 : -INFINITY;
                ps[hh * NK + row] = sc;
                mloc[hh] = fmaxf(mloc[hh], sc);
            }
        }
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        float v = mloc[hh];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0) red_m[hh * NW + warp] = v;
    }
    __syncthreads();
    // p = 2^(s - m) in place (n >= 1, so the chunk max m is finite) and row sums.
    float mh[G], lloc[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        float v = red_m[hh * NW];
#pragma unroll
        for (int w = 1; w < NW; ++w) v = fmaxf(v, red_m[hh * NW + w]);
        mh[hh] = v;
        lloc[hh] = 0.f;
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
        for (int t = tid; t < NK; t += kDecThreads) {
            const float p = t < n ? exp2f(ps[hh * NK + t] - mh[hh]) : 0.f;
            ps[hh * NK + t] = p;
            lloc[hh] += p;
        }
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        float v = lloc[hh];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red_l[hh * NW + warp] = v;
    }
    __syncthreads();
    // o_h = sum_t p_h(t) v_t: the same row groups; a v row is applied to all G heads.
    float acc[G][8];
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[hh][e] = 0.f;
#pragma unroll 4
    for (int st = 0; st < STEPS; ++st) {
        const int row = (st * NW + warp) * RPW + rl;
        if (row < n) {                                // rows past n hold no data
            const uint4 w = *reinterpret_cast<const uint4*>(sm + Sm::kV + row * DH * 2 + cl * 16);
            const float v8[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                                 bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const float p = ps[hh * NK + row];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[hh][e] = fmaf(p, v8[e], acc[hh][e]);
            }
        }
    }
    // lanes cl, cl + CPR, ... hold the same columns of different rows
#pragma unroll
    for (int off = CPR; off < 32; off <<= 1)
#pragma unroll
        for (int hh = 0; hh < G; ++hh)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[hh][e] += __shfl_xor_sync(0xffffffffu, acc[hh][e], off);
    if (rl == 0) {
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            float* d = osum + (warp * G + hh) * DH + cl * 8;
            *reinterpret_cast<float4*>(d) = make_float4(acc[hh][0], acc[hh][1], acc[hh][2], acc[hh][3]);
            *reinterpret_cast<float4*>(d + 4) = make_float4(acc[hh][4], acc[hh][5], acc[hh][6], acc[hh][7]);
        }
    }
    __syncthreads();
    if (ws / NK == pos / NK) {
        // All attended keys in this one chunk: the normalised output directly
        // (the combining launch sees a single chunk and does nothing).
        for (int i = tid; i < G * DH; i += kDecThreads) {
            const int hh = i / DH, d = i - hh * DH;
            float v = 0.f, l = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                v += osum[(w * G + hh) * DH + d];
                l += red_l[hh * NW + w];
            }
            o[(int64_t)(b * H + h0 + hh) * DH + d] = __float2bfloat16_rn(v / l);
        }
        return;
    }
    for (int i = tid; i < G * DH; i += kDecThreads) {
        const int hh = i / DH, d = i - hh * DH;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) v += osum[(w * G + hh) * DH + d];
        part[((int64_t)(b * H + h0 + hh) * nch + c) * (DH + 2) + d] = v;
    }
    if (tid < G) {
        float l = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) l += red_l[tid * NW + w];
        float m = mh[0];
#pragma unroll
        for (int hh = 1; hh < G; ++hh)
            if (hh == tid) m = mh[hh];                // mh[tid] with constant indices
        float* dst = part + ((int64_t)(b * H + h0 + tid) * nch + c) * (DH + 2);
        dst[DH] = m;
        dst[DH + 1] = l;
    }
}

// One CTA per (sequence, head) combines the chunks and writes o[b, h*DH + d]
// bf16: warp w owns columns [32 w, 32 w + 32), lane c takes chunk c0 + c (and
// c0 + c + 32, ...), so each chunk's max, sum and 32 columns are requested
// together and the combine costs one L2 round trip; the lanes' weighted column
// vectors are then summed through shared memory.
template <int DH>
__global__ void __launch_bounds__(DH) k_decode_combine(const float* __restrict__ part,
                                                      __nv_bfloat16* __restrict__ o, int BH,
                                                      int H, int nch_stride,
                                                      const int* __restrict__ pos_dev,
                                                      int window) {
    __shared__ float red[DH / 32][32][33];           // [warp][lane][column], padded
    pdl_wait();
    pdl_trigger();
    const int w = (int)blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (w >= BH) return;
    constexpr int NK = dec_keys(DH);
    const int pos = __ldg(pos_dev);
    const int nch = (pos + NK) / NK;                 // chunks holding keys [0, pos]
    const int ws = (window > 0 && pos - window + 1 > 0) ? pos - window + 1 : 0;
    const int c0 = ws / NK;                          // the first chunk in the window
    if (nch - c0 == 1) return;                       // written by the chunk kernel itself
    const float* p = part + (int64_t)w * nch_stride * (DH + 2);
    float M = -INFINITY, L = 0.f;
    float acc[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = 0.f;
    for (int cb = c0; cb < nch; cb += 32) {
        const int c = cb + lane;
        const bool has = c < nch;
        const float* pc = p + (int64_t)(has ? c : c0) * (DH + 2);
        const float mc = has ? pc[DH] : -INFINITY;
        const float lc = has ? pc[DH + 1] : 0.f;
        // a chunk's record is DH + 2 floats (even, so 8-byte aligned, not 16)
        float2 v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            v[j] = has ? *reinterpret_cast<const float2*>(pc + 32 * warp + 2 * j)
                       : make_float2(0.f, 0.f);
        // running max over the chunks seen so far (all lanes), rescaling what
        // earlier groups of 32 chunks accumulated
        float mb = mc;
#pragma unroll
        for (int s2 = 16; s2 > 0; s2 >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, s2));
        const float Mn = fmaxf(M, mb);
        const float keep = M == -INFINITY ? 0.f : exp2f(M - Mn);
        const float wgt = has ? exp2f(mc - Mn) : 0.f;
        L = L * keep + wgt * lc;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            acc[2 * j] = acc[2 * j] * keep + wgt * v[j].x;
            acc[2 * j + 1] = acc[2 * j + 1] * keep + wgt * v[j].y;
        }
        M = Mn;
    }
#pragma unroll
    for (int s2 = 16; s2 > 0; s2 >>= 1) L += __shfl_xor_sync(0xffffffffu, L, s2);
#pragma unroll
    for (int j = 0; j < 32; ++j) red[warp][lane][j] = acc[j];
    __syncwarp();
    float t = 0.f;
#pragma unroll 8
    for (int r = 0; r < 32; ++r) t += red[warp][r][lane];
    const int b = w / H, h = w - b * H;
    o[(int64_t)b * H * DH + (int64_t)h * DH + 32 * warp + lane] = __float2bfloat16_rn(t / L);
}

template <int DH, int G>
cudaError_t decode_launch(const void* q, const void* kc, const void* vc, float* part, void* o,
                          int B, int H, int Hkv, int max_seq, const int* pos_dev, float scale,
                          int window, cudaStream_t st) {
    // chunks for the longest possible cache; those past the length return at once
    using Sm = DecSmem<DH, G>;
    static bool attr_set = false;   // per instantiation; set once per process
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_decode_partial<DH, G>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Sm::kBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int nch = (max_seq + Sm::kKeys - 1) / Sm::kKeys;
    cudaError_t e = launch_pdl(k_decode_partial<DH, G>, dim3((unsigned)(B * Hkv * nch)),
                               dim3(kDecThreads), Sm::kBytes, st, static_cast<const __nv_bfloat16*>(q),
                               static_cast<const __nv_bfloat16*>(kc),
                               static_cast<const __nv_bfloat16*>(vc), part,
                               static_cast<__nv_bfloat16*>(o), H, Hkv, max_seq,
                               pos_dev, nch, scale * 1.4426950408889634f, window,
                               device_error_word());
    if (e != cudaSuccess) return e;
    const int BH = B * H;
    return launch_pdl(k_decode_combine<DH>, dim3((unsigned)BH), dim3(DH), 0, st,
                      static_cast<const float*>(part), static_cast<__nv_bfloat16*>(o), BH, H, nch,
                      pos_dev, window);
}

// Start of a decode step: the step's position and its B tokens go to device
// words that the recorded step reads, so the step itself has fixed arguments.
__global__ void k_decode_setup(int* pos_dev, int pos, const int32_t* tok, int32_t* tok_dev, int B) {
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0) *pos_dev = pos;
    for (int b = threadIdx.x; b < B; b += blockDim.x) tok_dev[b] = tok[b];
}

template <int DH>
cudaError_t decode_dh(const void* q, const void* kc, const void* vc, float* part, void* o, int B,
                      int H, int Hkv, int max_seq, const int* L, float scale, int window,
                      cudaStream_t st) {
    switch (H / Hkv) {
        case 1: return decode_launch<DH, 1>(q, kc, vc, part, o, B, H, Hkv, max_seq, L, scale, window, st);
        case 2: return decode_launch<DH, 2>(q, kc, vc, part, o, B, H, Hkv, max_seq, L, scale, window, st);
        case 4: return decode_launch<DH, 4>(q, kc, vc, part, o, B, H, Hkv, max_seq, L, scale, window, st);
        case 8: return decode_launch<DH, 8>(q, kc, vc, part, o, B, H, Hkv, max_seq, L, scale, window, st);
        case 16:
            // 16 heads of 128 columns would need 57.6 KB of static shared memory
            if constexpr (DH <= 64)
                return decode_launch<DH, 16>(q, kc, vc, part, o, B, H, Hkv, max_seq, L, scale, window, st);
            return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t decode_partial_floats(int B, int H, int max_seq, int dh) {
    const int nk = dec_keys(dh);
    return (size_t)B * H * ((max_seq + nk - 1) / nk) * (dh + 2);
}

bool decode_supported(int dh, int group) {
    return (dh == 32 || dh == 64 || dh == 128) &&
           (group == 1 || group == 2 || group == 4 || group == 8 || (group == 16 && dh <= 64));
}

cudaError_t launch_decode_attention(const void* q, const void* kc, const void* vc, float* part,
                                    void* o, int B, int H, int Hkv, int max_seq,
                                    const int* L, int dh, float scale, cudaStream_t st,
                                    int window) {
    if (B <= 0) return cudaSuccess;
    switch (dh) {
        case 32: return decode_dh<32>(q, kc, vc, part, o, B, H, Hkv, max_seq, L, scale, window, st);
        case 64: return decode_dh<64>(q, kc, vc, part, o, B, H, Hkv, max_seq, L, scale, window, st);
        case 128: return decode_dh<128>(q, kc, vc, part, o, B, H, Hkv, max_seq, L, scale, window, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode_setup(int* pos_dev, int pos, const int32_t* tok, int32_t* tok_dev, int B,
                                cudaStream_t st) {
    return launch_pdl(k_decode_setup, dim3(1), dim3(256), 0, st, pos_dev, pos, tok, tok_dev, B);
}

}  // namespace tfm
