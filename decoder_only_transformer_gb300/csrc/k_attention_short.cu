// k_attention_short.cu - causal softmax attention on tcgen05 for d_head 32 and
// sequences of at most 256 positions.
//
// Same mathematics as the other attention kernels (CS336 walkthrough, section
// 5.4; "LLM 2", section GQA / MQA): o = softmax(q k^T / sqrt(dh) + M) v with
// M = -inf above the diagonal, kv head = h / (H / Hkv).  Here a whole
// (sequence, head) fits at once.  With query and key tiles A = [0, 128) and
// B = [128, 256), the causal product has three 128 x 128 blocks:
//   block 0: queries A, keys A (diagonal)
//   block 1: queries B, keys A (no mask)
//   block 2: queries B, keys B (diagonal)
// Each block has its own softmax warpgroup, tensor-memory columns and output
// accumulator, so the three run side by side: the critical path of an item is
// one block, not the two key tiles of query tile B in a row.  Block 1 and block
// 2 each keep their own row max and sum; query tile B's output is their exact
// merge, o = (O1 2^(m1-m) + O2 2^(m2-m)) / (l1 2^(m1-m) + l2 2^(m2-m)) with
// m = max(m1, m2), done once per item (the split-K form of flash decoding).
//
// One CTA of 16 warps per SM, persistent over (sequence, head) items:
//   warp 0      TMA: Q, K and V of an item (six 128 x 32 boxes, 48 KB) into one
//               of three buffers, so the next items' loads run ahead
//   warps 4-7, 8-11, 12-15  blocks 0, 1, 2, one thread per query row.  Each
//               warpgroup drives its own block: its first thread issues the S
//               product (M = N = 128, K = 32) and, once all four warps have
//               written P (a bounded mbarrier), the P.V product (P from tensor memory, V MN-major,
//               M = 128, N = 32, K = 128); the next item's S is issued as soon
//               as this item's P.V is done, so it runs under the output readout.
//               The softmax takes the row max over the block's S columns, then
//               computes p = 2^(s scale log2e - m), sums it and writes it back as
//               bf16 pairs over the S columns already read.  Warps 4-7 write
//               query tile A's output rows, warps 8-11 hand block 1's rows to
//               warps 12-15 through shared memory, which merge and write tile B's.
// (A separate MMA-issuing warp was measured to be the bound: sharing its
// scheduler with busy softmax warps it took ~1000 cycles to issue a block's
// eight P.V products, against a ~2500-cycle softmax.)
// Chunks of 32 keys that lie wholly above a block's diagonal, or past the
// sequence, are skipped (their p are written as 0).  Every wait is bounded.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace tfm {

namespace {

constexpr int kDH = 32;
constexpr int kT = 128;                           // query and key tile
constexpr int kThreadsShort = 512;
constexpr int kBufs = 3;                          // item buffers in shared memory
constexpr int kBoxBytes = kT * kDH * 2;           // one 128 x 32 bf16 box, 64-byte rows
constexpr int kBufBytes = 6 * kBoxBytes;          // Q_A, Q_B, K_A, K_B, V_A, V_B
// Block 1's output handed to block 2's merge: per slot (item parity) the 32
// unnormalised values of each row stored column-major ([e][row], conflict-free
// for a warp), then the rows' (max, sum).
constexpr int kHandFloats = kDH * kT + 2 * kT;
constexpr int kHandOff = kBufs * kBufBytes;
constexpr int kBarOff = kHandOff + 2 * kHandFloats * 4;
// full[3], empty[3], s_full[3], o_done[3], p_ready[3], hand_full[2], hand_free[2]
constexpr int kNumBars = 2 * kBufs + 3 * 3 + 4;
constexpr int kMiscOff = kBarOff + 8 * kNumBars;
constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + alignment slack
constexpr int kOCol = 3 * kT;                     // O_x at tensor-memory column 384 + 32 x
constexpr uint32_t kSwz64 = 4u;                   // 64-byte swizzle (descriptor code)
constexpr uint32_t kGroup = 8 * kDH * 2;          // 8-row swizzle atom, 512 bytes

__global__ void __launch_bounds__(kThreadsShort, 1)
    k_attention_short(const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, __nv_bfloat16* __restrict__ o,
                      int BH, int H, int Hkv, int S, float scale_log2, int* err) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t bars = base + kBarOff;
    auto full_bar = [&](int b) { return bars + 8u * b; };
    auto empty_bar = [&](int b) { return bars + 8u * (kBufs + b); };
    auto s_full = [&](int x) { return bars + 8u * (2 * kBufs + x); };
    auto o_done = [&](int x) { return bars + 8u * (2 * kBufs + 3 + x); };
    auto p_ready = [&](int x) { return bars + 8u * (2 * kBufs + 6 + x); };
    auto hand_full = [&](int sl) { return bars + 8u * (2 * kBufs + 9 + sl); };
    auto hand_free = [&](int sl) { return bars + 8u * (2 * kBufs + 11 + sl); };
    float* hand = reinterpret_cast<float*>(gbase + kHandOff);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(gbase + kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kMiscOff + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool has_b = S > kT;
    const int nblk = has_b ? 3 : 1;
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    const int items = (BH - c + G - 1) / G;           // items c, c + G, ... of this CTA
    const int group = H / Hkv;

    if (warp == 0 && lane == 0) {
        for (int b = 0; b < kBufs; ++b) {
            mbar_init(full_bar(b), 1);
            mbar_init(empty_bar(b), nblk);             // each block's last product releases it
        }
        for (int x = 0; x < 3; ++x) {
            mbar_init(s_full(x), 1);
            mbar_init(o_done(x), 1);
            mbar_init(p_ready(x), 4);
        }
        for (int sl = 0; sl < 2; ++sl) {
            mbar_init(hand_full(sl), 4);
            mbar_init(hand_free(sl), 4);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&qmap);
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_holder), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            const uint32_t bytes = (uint32_t)(has_b ? 6 : 3) * kBoxBytes;
            int issued = 0;
            for (int i = 0; i < items; ++i) {
                const int bh = c + i * G;
                const int b = bh / H, h = bh - b * H, g = h / group;
                const int buf = i % kBufs;
                if (i >= kBufs &&
                    !mbar_wait(empty_bar(buf), (uint32_t)(i / kBufs - 1) & 1u, err, abort_flag))
                    break;
                const uint32_t sb = base + buf * kBufBytes;
                mbar_arrive_expect_tx(full_bar(buf), bytes);
                tma_load_3d(sb, &qmap, 0, 0, b * H + h, full_bar(buf));
                tma_load_3d(sb + 2 * kBoxBytes, &kmap, 0, 0, b * Hkv + g, full_bar(buf));
                tma_load_3d(sb + 4 * kBoxBytes, &vmap, 0, 0, b * Hkv + g, full_bar(buf));
                if (has_b) {
                    tma_load_3d(sb + kBoxBytes, &qmap, 0, kT, b * H + h, full_bar(buf));
                    tma_load_3d(sb + 3 * kBoxBytes, &kmap, 0, kT, b * Hkv + g, full_bar(buf));
                    tma_load_3d(sb + 5 * kBoxBytes, &vmap, 0, kT, b * Hkv + g, full_bar(buf));
                }
                ++issued;
            }
            // No copy may be in flight when the CTA ends.
            for (int i = issued - kBufs < 0 ? 0 : issued - kBufs; i < issued; ++i)
                mbar_wait(full_bar(i % kBufs), (uint32_t)(i / kBufs) & 1u, err, abort_flag);
        }
    } else if (warp >= 4 && (warp - 4) / 4 < nblk) {
        // ---------------------------------------------------------- blocks
        const int x = (warp - 4) >> 2;                 // block of this warpgroup
        const int q4 = warp & 3;                       // TMEM lane quarter
        const int r = q4 * 32 + lane;                  // row inside the query tile
        const bool issuer = q4 == 0 && lane == 0;      // issues this block's products
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const uint32_t t_s = tmem_base + x * kT + lane_off;
        const uint32_t t_o = tmem_base + kOCol + x * kDH + lane_off;
        const bool diag = x != 1;
        const int q0 = x == 0 ? 0 : kT;                // first query of the tile
        const int k0 = x == 2 ? kT : 0;                // first key of the block
        const int qi = q0 + r;
        // Keys [0, kend) of the block are visible to this row: before the end of
        // the sequence and, on a diagonal block, not after the query.
        int kend = S - k0 < kT ? S - k0 : kT;
        if (diag && r + 1 < kend) kend = r + 1;
        // Chunks this warp needs at all (those of any of its rows); chunks below
        // kfull are visible to every row of the warp.
        int wend = S - k0 < kT ? S - k0 : kT;
        if (diag && q4 * 32 + 32 < wend) wend = q4 * 32 + 32;
        const int nck = wend > 0 ? (wend + 31) / 32 : 0;
        const int kfull = __reduce_min_sync(0xffffffffu, kend < 0 ? 0 : kend);
        constexpr uint32_t idesc_s = umma_idesc_bf16(kT, kT);
        constexpr uint32_t idesc_o = umma_idesc_bf16(kT, kDH, true);
        const uint64_t dq = sdesc(base, kSwz64, 16, kGroup);
        const uint64_t dv = sdesc(base, kSwz64, 0, kGroup);
        const int qbox = x == 0 ? 0 : 1, kbox = x == 2 ? 3 : 2, vbox = x == 2 ? 5 : 4;
        // S_x of item i (the issuer; P_x of item i - 1, written over S_x, has been
        // consumed: its P.V is complete).
        auto issue_s = [&](int i) -> bool {
            const int buf = i % kBufs;
            if (!mbar_wait(full_bar(buf), (uint32_t)(i / kBufs) & 1u, err, abort_flag)) return false;
            tc_fence_after();
            const uint64_t a0 = dq + (uint64_t)((buf * kBufBytes + qbox * kBoxBytes) >> 4);
            const uint64_t b0 = dq + (uint64_t)((buf * kBufBytes + kbox * kBoxBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < kDH / 16; ++kk)
                umma_bf16(tmem_base + x * kT, a0 + 2 * kk, b0 + 2 * kk, idesc_s, kk > 0 ? 1u : 0u);
            umma_commit(s_full(x));
            return true;
        };
        bool ok = true;
        if (issuer && items > 0) ok = issue_s(0);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        for (int i = 0; i < items && ok; ++i) {
            const int bh = c + i * G;
            const int b = bh / H, h = bh - b * H;
            const int buf = i % kBufs;
            if (!warp_wait(s_full(x), (uint32_t)i & 1u, err, abort_flag)) { ok = false; break; }
            tc_fence_after();
            // Pass 1: the row max over the visible keys.
            float mx = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < kT / 32; ++cc) {
                if (cc >= nck) break;
                float v[32];
                tmem_ld32(t_s + cc * 32, v);
                if ((cc + 1) * 32 > kfull) {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (cc * 32 + e >= kend) v[e] = -INFINITY;
                }
                // two chains of three-input maxima over v[0..31]
                float ma = fmax3(v[0], v[1], v[2]), mb = fmax3(v[3], v[4], v[5]);
#pragma unroll
                for (int e = 6; e < 30; e += 4) {
                    ma = fmax3(ma, v[e], v[e + 1]);
                    mb = fmax3(mb, v[e + 2], v[e + 3]);
                }
                ma = fmax3(ma, v[30], v[31]);
                mx = fmax3(mx, ma, mb);
            }
            const float m = mx * scale_log2;
            // (a row with no visible key, past the sequence: p = 0, never written out)
            const float negm = m == -INFINITY ? 0.f : -m;
            // Pass 2: p = 2^(s scale - m), row sum, P over the consumed S columns
            // (keys 32 cc .. 32 cc + 31 -> columns 16 cc .. 16 cc + 15).  Chunk
            // cc + 1's load is in flight while chunk cc is computed; every
            // destination of a load stays live until its wait.
            const uint64_t scale2 = f2_pack(scale_log2, scale_log2);
            const uint64_t negm2 = f2_pack(negm, negm);
            uint64_t sum2[2] = {0ull, 0ull};
            uint32_t cur[32];
            if (nck > 0) {
                tmem_ld32_issue(t_s, cur);
                tmem_ld_wait();
                reg_fence32(cur);
            }
#pragma unroll
            for (int cc = 0; cc < kT / 32; ++cc) {
                uint32_t pw[16];
                if (cc < nck) {
                    uint32_t nxt[32];
                    const bool more = cc + 1 < nck;
                    if (more) tmem_ld32_issue(t_s + (cc + 1) * 32, nxt);
                    const bool masked = (cc + 1) * 32 > kfull;
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float t0, t1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(cur[e]), __uint_as_float(cur[e + 1])),
                                         scale2, negm2),
                                  t0, t1);
                        float p0 = fast_exp2(t0), p1 = fast_exp2(t1);
                        if (masked) {
                            if (cc * 32 + e >= kend) p0 = 0.f;
                            if (cc * 32 + e + 1 >= kend) p1 = 0.f;
                        }
                        sum2[(e >> 1) & 1] = f2_add(sum2[(e >> 1) & 1], f2_pack(p0, p1));
                        pw[e >> 1] = pack_bf16x2(p0, p1);
                    }
                    if (more) {
                        tmem_ld_wait();
                        reg_fence32(nxt);
#pragma unroll
                        for (int e = 0; e < 32; ++e) cur[e] = nxt[e];
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) pw[e] = 0u;
                }
                tmem_st16_async(t_s + cc * 16, pw);
            }
            tmem_st_wait();
            float sa[2], sb[2];
            f2_unpack(sum2[0], sa[0], sb[0]);
            f2_unpack(sum2[1], sa[1], sb[1]);
            const float l = (sa[0] + sb[0]) + (sa[1] + sb[1]);
            // Once P_x is complete in all four lane quarters (p_ready), the issuer
            // starts P_x.V; a second commit releases the item's buffer when this
            // block's products of the item are done.
            bool nok_p = true;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_ready(x));
            if (issuer) {
                if (!mbar_wait(p_ready(x), (uint32_t)i & 1u, err, abort_flag)) nok_p = false;
            }
            if (!__shfl_sync(0xffffffffu, nok_p ? 1 : 0, 0)) { ok = false; break; }
            if (issuer) {
                tc_fence_after();
                const uint64_t b0 = dv + (uint64_t)((buf * kBufBytes + vbox * kBoxBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < kT / 16; ++kk)
                    umma_bf16_ts(tmem_base + kOCol + x * kDH, tmem_base + x * kT + kk * 8,
                                 b0 + kk * ((16 * kDH * 2) >> 4), idesc_o, kk > 0 ? 1u : 0u);
                umma_commit(o_done(x));
                umma_commit(empty_bar(buf));
            }
            if (!warp_wait(o_done(x), (uint32_t)i & 1u, err, abort_flag)) { ok = false; break; }
            tc_fence_after();
            // P_x is consumed: the next item's S_x runs under this item's readout.
            bool nok = true;
            if (issuer && i + 1 < items) nok = issue_s(i + 1);
            if (!__shfl_sync(0xffffffffu, nok ? 1 : 0, 0)) { ok = false; break; }
            const int sl = i & 1;
            float* hs = hand + sl * kHandFloats;
            float ov[32];
            tmem_ld32(t_o, ov);
            if (x == 1) {
                // Block 1: the unnormalised rows and their (max, sum) go to the
                // merge of warps 12-15 through shared memory (slot i % 2, rewritten
                // after the merge of item i - 2).
                if (i >= 2 && !warp_wait(hand_free(sl), (uint32_t)((i >> 1) - 1) & 1u, err, abort_flag)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int e = 0; e < 32; ++e) hs[e * kT + r] = ov[e];
                hs[kDH * kT + 2 * r] = m;
                hs[kDH * kT + 2 * r + 1] = l;
                __syncwarp();
                if (lane == 0) mbar_arrive(hand_full(sl));
                continue;
            }
            float inv;
            if (x == 0) {
                inv = 1.0f / l;
            } else {
                // exact merge with block 1 (same rows, its own max and sum)
                if (!warp_wait(hand_full(sl), (uint32_t)(i >> 1) & 1u, err, abort_flag)) {
                    ok = false;
                    break;
                }
                const float m1 = hs[kDH * kT + 2 * r], l1 = hs[kDH * kT + 2 * r + 1];
                const float mm = fmaxf(m1, m);
                const float a1 = fast_exp2(m1 - mm), a2 = fast_exp2(m - mm);
                inv = 1.0f / (l1 * a1 + l * a2);
#pragma unroll
                for (int e = 0; e < 32; ++e) ov[e] = hs[e * kT + r] * a1 + ov[e] * a2;
                __syncwarp();
                if (lane == 0) mbar_arrive(hand_free(sl));
            }
            if (qi < S) {
                __nv_bfloat16* orow = o + ((int64_t)(b * S + qi) * H + h) * kDH;
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    uint4 w;
                    w.x = pack_bf16x2(ov[e] * inv, ov[e + 1] * inv);
                    w.y = pack_bf16x2(ov[e + 2] * inv, ov[e + 3] * inv);
                    w.z = pack_bf16x2(ov[e + 4] * inv, ov[e + 5] * inv);
                    w.w = pack_bf16x2(ov[e + 6] * inv, ov[e + 7] * inv);
                    *reinterpret_cast<uint4*>(orow + e) = w;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

}  // namespace

bool attention_short_supported(int dh, int S, int window) {
    return dh == kDH && S > 0 && S <= 2 * kT && window == 0;
}

cudaError_t launch_attention_short(const AttnPlan& p, cudaStream_t st) {
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    if (p.B <= 0 || p.S <= 0) return cudaSuccess;
    if (!attention_short_supported(p.dh, p.S, p.window)) return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_attention_short,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    // One CTA per SM (shared memory and tensor memory allow no more).
    const int bh = p.B * p.H;
    const int grid = bh < sm_count() ? bh : sm_count();
    return launch_pdl(k_attention_short, dim3(grid), dim3(kThreadsShort), kSmemBytes, st, p.qmap,
                      p.kmap, p.vmap, static_cast<__nv_bfloat16*>(p.o), bh, p.H, p.Hkv, p.S,
                      p.scale * 1.4426950408889634f, device_error_word());
}

}  // namespace tfm
