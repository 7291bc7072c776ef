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
//   warp 1      S MMAs: S_x = Q K^T into 128 TMEM columns per block (M = N = 128,
//               K = 32)
//   warp 2      P.V MMAs: O_x = P_x V, P read from tensor memory, V MN-major
//               (M = 128, N = 32, K = 128)
//   warps 4-7, 8-11, 12-15  softmax of blocks 0, 1, 2, one thread per query row:
//               a first pass over the block's S columns takes the row max, a
//               second computes p = 2^(s scale log2e - m), sums it and writes it
//               back as bf16 pairs over the S columns already read; warps 4-7
//               then write query tile A's output rows, warps 12-15 merge blocks 1
//               and 2 (block 1's output read from tensor memory, its max and sum
//               from shared memory) and write tile B's.
// Chunks of 32 keys that lie wholly above a block's diagonal, or past the
// sequence, are skipped (their p are written as 0).  Every wait is bounded.
//
// Measured at the short-sequence workload (32 x 256 positions, 16 heads): 19.1
// us against 21.0 us for an mma.sync flash kernel.  A per-CTA clock-stamp
// timeline gives ~5500 cycles per item: ~450 from issuing S to the softmax
// seeing it, ~700 for the max pass, ~2500 for the exponential pass, ~1000 from
// P to the end of P.V (the three blocks' 24 P.V products, N = 32, share the
// tensor pipe at about a third of its rate).  Tensor memory (480 of 512
// columns) allows no second item in flight.  Two reorganisations measured
// slower (21.7 us): issuer warps that poll every block's barriers and issue
// whichever is ready, with block 1's output handed over through shared memory;
// and warpgroups that issue their own products.  Also measured against this
// kernel on one box (per-CTA clock stamps, 13.3 us for the whole launch with q,
// k, v in L2), none kept:
//   - tile A's 32-row groups loaded in reverse order, so that the heavy rows of
//     the two diagonal blocks fall on different schedulers: 14.3 us.  Block 2
//     runs about one step of the pipeline behind blocks 0 and 1, so the two
//     triangles never overlap and the reversal only moves the heavy scheduler.
//   - P handed to the P.V issuer 32 keys at a time, so that the products run
//     under the exponentials: 15-20 us.  The issuing thread gets about a quarter
//     of its scheduler's issue slots, and per-chunk waits and fences on it delay
//     every block's output; a second issuer for block 1 (15-16.5 us) and polling
//     with a short sleep (no change) did not recover it.
//   - the masking test written per score as (diagonal chunk and column past the
//     row) or (column past the sequence): the exponential pass took twice as
//     long as with one precomputed threshold per chunk.  Every instruction per
//     score counts in that loop.
//   - P in shared memory (128-byte swizzled, the A operand of P.V) instead of
//     over S, so that the next item's S_x is issued as soon as the softmax has
//     read S_x: 13.7-14.7 us with two item buffers (the shared-memory budget),
//     also with Q/K and V released separately and with the reversed groups.
//     The three blocks then run side by side and each exponential pass slows
//     down as much as the chain got shorter.
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
constexpr int kBarOff = kBufs * kBufBytes;
// full[3], empty[3], s_full[3], p_full[3], o_done[3], o_free[3], stats, done
constexpr int kNumBars = 2 * kBufs + 5 * 3 + 2;
constexpr int kStatsOff = kBarOff + 8 * kNumBars; // (m, l) of block 1 rows, two items
constexpr int kMiscOff = kStatsOff + 2 * kT * 8;
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
    auto p_full = [&](int x) { return bars + 8u * (2 * kBufs + 3 + x); };
    auto o_done = [&](int x) { return bars + 8u * (2 * kBufs + 6 + x); };
    auto o_free = [&](int x) { return bars + 8u * (2 * kBufs + 9 + x); };
    const uint32_t stats_bar = bars + 8u * (2 * kBufs + 12);
    const uint32_t done_bar = bars + 8u * (2 * kBufs + 13);
    float2* stats = reinterpret_cast<float2*>(gbase + kStatsOff);
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
            mbar_init(empty_bar(b), 2);                // both MMA issuers release a buffer
        }
        for (int x = 0; x < 3; ++x) {
            mbar_init(s_full(x), 1);
            mbar_init(p_full(x), 4);
            mbar_init(o_done(x), 1);
            mbar_init(o_free(x), 4);
        }
        mbar_init(stats_bar, 4);
        mbar_init(done_bar, 2);
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
    } else if (warp == 1) {
        // ---------------------------------------------------------- S issuer
        // Releases an item's buffer (with the P.V issuer) by a commit after its
        // last product reading it; both commit to done_bar at the end, so no
        // product is in flight when tensor memory is freed.
        if (lane == 0) {
            bool ok = true;
            constexpr uint32_t idesc_s = umma_idesc_bf16(kT, kT);
            const uint64_t d0 = sdesc(base, kSwz64, 16, kGroup);
            for (int i = 0; i < items && ok; ++i) {
                const int buf = i % kBufs;
                ok = mbar_wait(full_bar(buf), (uint32_t)(i / kBufs) & 1u, err, abort_flag);
                for (int x = 0; x < nblk && ok; ++x) {
                    // P_x is written over S_x: the next S_x waits for the last P_x.V
                    if (i > 0) ok = mbar_wait(o_done(x), (uint32_t)(i - 1) & 1u, err, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    const int qbox = x == 0 ? 0 : 1, kbox = x == 2 ? 3 : 2;
                    const uint64_t a0 = d0 + (uint64_t)((buf * kBufBytes + qbox * kBoxBytes) >> 4);
                    const uint64_t b0 = d0 + (uint64_t)((buf * kBufBytes + kbox * kBoxBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kDH / 16; ++kk)
                        umma_bf16(tmem_base + x * kT, a0 + 2 * kk, b0 + 2 * kk, idesc_s, kk > 0 ? 1u : 0u);
                    umma_commit(s_full(x));
                }
                if (ok) umma_commit(empty_bar(buf));
            }
            umma_commit(done_bar);
            mbar_wait(done_bar, 0, err, abort_flag);
        }
    } else if (warp == 2) {
        // ---------------------------------------------------------- P.V issuer
        if (lane == 0) {
            bool ok = true;
            constexpr uint32_t idesc_o = umma_idesc_bf16(kT, kDH, true);
            const uint64_t dv = sdesc(base, kSwz64, 0, kGroup);
            for (int i = 0; i < items && ok; ++i) {
                const int buf = i % kBufs;
                for (int x = 0; x < nblk && ok; ++x) {
                    ok = mbar_wait(p_full(x), (uint32_t)i & 1u, err, abort_flag);
                    // O_x is overwritten once the previous item's O_x has been read
                    if (ok && i > 0) ok = mbar_wait(o_free(x), (uint32_t)(i - 1) & 1u, err, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    const int vbox = x == 2 ? 5 : 4;
                    const uint64_t b0 = dv + (uint64_t)((buf * kBufBytes + vbox * kBoxBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kT / 16; ++kk)
                        umma_bf16_ts(tmem_base + kOCol + x * kDH, tmem_base + x * kT + kk * 8,
                                     b0 + kk * ((16 * kDH * 2) >> 4), idesc_o, kk > 0 ? 1u : 0u);
                    umma_commit(o_done(x));
                }
                if (ok) umma_commit(empty_bar(buf));
            }
            umma_commit(done_bar);
            mbar_wait(done_bar, 0, err, abort_flag);
        }
    } else if (warp >= 4 && (warp - 4) / 4 < nblk) {
        // ---------------------------------------------------------- softmax
        const int x = (warp - 4) >> 2;                 // block of this warpgroup
        const int q4 = warp & 3;                       // TMEM lane quarter
        const int r = q4 * 32 + lane;                  // row inside the query tile
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
        bool ok = true;
        for (int i = 0; i < items && ok; ++i) {
            const int bh = c + i * G;
            const int b = bh / H, h = bh - b * H;
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
            // (keys 32 cc .. 32 cc + 31 -> columns 16 cc .. 16 cc + 15).
            const uint64_t scale2 = f2_pack(scale_log2, scale_log2);
            const uint64_t negm2 = f2_pack(negm, negm);
            uint64_t sum2[2] = {0ull, 0ull};
#pragma unroll
            for (int cc = 0; cc < kT / 32; ++cc) {
                uint32_t pw[16];
                if (cc < nck) {
                    float v[32];
                    tmem_ld32(t_s + cc * 32, v);
                    const bool masked = (cc + 1) * 32 > kfull;
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float t0, t1;
                        f2_unpack(f2_fma(f2_pack(v[e], v[e + 1]), scale2, negm2), t0, t1);
                        float p0 = fast_exp2(t0), p1 = fast_exp2(t1);
                        if (masked) {
                            if (cc * 32 + e >= kend) p0 = 0.f;
                            if (cc * 32 + e + 1 >= kend) p1 = 0.f;
                        }
                        sum2[(e >> 1) & 1] = f2_add(sum2[(e >> 1) & 1], f2_pack(p0, p1));
                        pw[e >> 1] = pack_bf16x2(p0, p1);
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
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(x));
            if (x == 1) {
                // Block 1 hands its (max, sum) to the merge of warps 12-15; the
                // slot of item i is rewritten only after item i - 2's merge.
                if (i > 0 && !warp_wait(o_free(1), (uint32_t)(i - 1) & 1u, err, abort_flag)) {
                    ok = false;
                    break;
                }
                stats[(i & 1) * kT + r] = make_float2(m, l);
                __syncwarp();
                if (lane == 0) mbar_arrive(stats_bar);
                continue;
            }
            // Blocks 0 and 2: wait for this block's P.V (block 2 also for block
            // 1's and its statistics), then write the output rows.
            bool got = warp_wait(o_done(x), (uint32_t)i & 1u, err, abort_flag);
            if (got && x == 2)
                got = warp_wait(o_done(1), (uint32_t)i & 1u, err, abort_flag) &&
                      warp_wait(stats_bar, (uint32_t)i & 1u, err, abort_flag);
            if (!got) { ok = false; break; }
            tc_fence_after();
            float ov[32];
            tmem_ld32(t_o, ov);
            float inv;
            if (x == 0) {
                inv = 1.0f / l;
            } else {
                // exact merge with block 1 (same rows, its own max and sum)
                float o1[32];
                tmem_ld32(tmem_base + kOCol + kDH + lane_off, o1);
                const float2 st = stats[(i & 1) * kT + r];
                const float mm = fmaxf(st.x, m);
                const float a1 = fast_exp2(st.x - mm), a2 = fast_exp2(m - mm);
                inv = 1.0f / (st.y * a1 + l * a2);
#pragma unroll
                for (int e = 0; e < 32; ++e) ov[e] = o1[e] * a1 + ov[e] * a2;
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
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(o_free(x));
                if (x == 2) mbar_arrive(o_free(1));
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
