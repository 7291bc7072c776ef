// k_attention_tc.cu - causal softmax attention on the sm_103a tensor cores
// (tcgen05 + tensor memory), d_head 128.
//
// o = softmax(q k^T * scale + M) v per (sequence, head), M = -inf above the
// diagonal (CS336 walkthrough, section 5.4), query head h reading kv head
// h / (H / Hkv) ("LLM 2", section GQA / MQA).  The softmax is evaluated online
// over key tiles: a running row max and row sum, the partial output rescaled
// when the max grows (stable softmax: subtracting any common constant leaves
// the result unchanged, so the rescale is exact up to rounding).
//
// A work item is 128 query rows of one (sequence, head), keys in tiles of 128.
// The kernel is persistent: one CTA per SM walks a list of items (longest first
// across all heads, dealt in snake order), and an item's tail overlaps the next
// item's start.  Measured per-item timelines showed why both matter: a CTA per
// item left the SMs idle ~30 % of the kernel between CTAs, and writing O out
// from the softmax warps stalled them ~4000 cycles per item (wait for the last
// P.V, read O, normalise, store 32 KB) against ~1400 cycles per key tile.
//   warp 0      TMA: each item's Q tile into one of two Q buffers (item parity;
//               refilled once the S MMAs of the item two back are done, so the
//               next item's Q arrives while this one runs), then K and V tiles
//               (3-D maps [seq*heads, S, dh], 128-byte swizzle, zero fill past S)
//               into a 2-deep K ring and a 3-deep V ring, in the order the MMA
//               threads consume them.  (With one Q buffer the next item's S had
//               to wait for this item's last S and then a TMA round trip: GQA
//               workload 61.2 -> 59.6 us with two; the second buffer took a K
//               ring slot, shared memory being full.)
//   warp 1      TMEM (512 columns: S double buffer 2 x 128, O dh, P double buffer
//               2 x 64) and the S MMAs: S_j = Q K_j^T (M=128, N=128, K=dh)
//   warp 2      the P.V MMAs: O += P_j V_j (M=128, N=dh, K=128; P read from tensor
//               memory, V read MN-major straight from its [key, dh] tile, so it is
//               never transposed); an item's first P.V (which overwrites O) waits
//               until the epilogue warps have read the previous item's O.
//               Issuing from two threads keeps the per-thread instruction stream
//               short: an MMA warp shares its scheduler with busy warps.
//   warp 3      idle (the control warps form one warpgroup)
//   warps 4..7  softmax, one thread per query row: S row from TMEM, causal /
//               length mask, row max, p = 2^(s*scale*log2e - m) stored as bf16
//               pairs into the P columns of tensor memory, row sum; the partial
//               O in TMEM is rescaled only when the row max grows by more than
//               2^8, so P entries stay below 256 and most tiles skip the rescale.
//               At the end of an item they hand the row sums to the epilogue
//               through shared memory and go on to the next item.
//   warps 8..11 epilogue: per item, after its last P.V, O out of tensor memory,
//               O / l as bf16 to global memory (heads merged).
// S_{j+1} runs on the tensor cores while the softmax warps work on S_j.
// Tiles entirely above the diagonal are never loaded.  All waits are bounded.
// (Taking an unmasked tile's row maximum from the tensor-memory load with
// tcgen05.ld.red, sm_103a, measured no different here: GQA workload 63.2 vs
// 63.4 us, so the maxima are not what bounds this softmax.)
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace tfm {

namespace {

constexpr int kQ = 128;
constexpr int kKV = 128;
constexpr int kThreadsAtt = 384;   // 4 control warps, 4 softmax warps, 4 epilogue warps
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <int DH>
struct AttTc {
    static constexpr int kStages = DH == 64 ? 4 : 3;  // V ring
    static constexpr int kKStages = DH == 64 ? 4 : 2; // K ring (the second Q buffer took a slot)
    static constexpr int kSub = DH / 64;              // 64-column (128-byte) sub-tiles
    static constexpr int kQBytes = kQ * DH * 2;
    static constexpr int kKBytes = kKV * DH * 2;
    static constexpr int kVBytes = kKV * DH * 2;
    static constexpr int kQOff = 0;                   // two Q buffers (item parity)
    static constexpr int kKOff = kQOff + 2 * kQBytes;
    static constexpr int kVOff = kKOff + kKStages * kKBytes;
    static constexpr int kBarOff = kVOff + kStages * kVBytes;
    static constexpr int kOCol = 2 * kKV;             // TMEM columns: S[2], O, P[2]
    static constexpr int kPCol = kOCol + DH;
    // k_full[SK], k_empty[SK], v_full[S], v_empty[S], s_full[2], p_full[2],
    // o_done[2], done, l_ready, o_free, q_full[2], q_empty[2]
    static constexpr int kNumBars = 2 * kKStages + 2 * kStages + 13;
    // Row sums handed from the softmax to the epilogue warps, [item parity][row].
    static constexpr int kRedOff = kBarOff + 8 * kNumBars;
    static constexpr int kMiscOff = kRedOff + 2 * kQ * 4;
    static constexpr int kBytes = kMiscOff + 16 + 1024;
};

template <int DH, bool kWin>
__global__ void __launch_bounds__(kThreadsAtt, 1)
    k_attention_tc(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, __nv_bfloat16* __restrict__ o, int BH,
                   int H, int Hkv, int S, float scale_log2, int window, int* err) {
    using L = AttTc<DH>;
    constexpr int ST = L::kStages, SK = L::kKStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t sQ = base + L::kQOff, sK = base + L::kKOff, sV = base + L::kVOff;
    const uint32_t bars = base + L::kBarOff;
    constexpr int B0 = 2 * SK + 2 * ST;               // first barrier after the rings
    auto k_full = [&](int s) { return bars + 8u * s; };
    auto k_empty = [&](int s) { return bars + 8u * (SK + s); };
    auto v_full = [&](int s) { return bars + 8u * (2 * SK + s); };
    auto v_empty = [&](int s) { return bars + 8u * (2 * SK + ST + s); };
    auto s_full = [&](int i) { return bars + 8u * (B0 + i); };
    auto p_full = [&](int i) { return bars + 8u * (B0 + 2 + i); };
    auto o_done = [&](int i) { return bars + 8u * (B0 + 4 + i); };
    const uint32_t done_bar = bars + 8u * (B0 + 6);
    const uint32_t l_ready = bars + 8u * (B0 + 7);
    const uint32_t o_free = bars + 8u * (B0 + 8);
    auto q_full = [&](int qb) { return bars + 8u * (B0 + 9 + qb); };
    auto q_empty = [&](int qb) { return bars + 8u * (B0 + 11 + qb); };
    float* red_l = reinterpret_cast<float*>(gbase + L::kRedOff);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(gbase + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_qt = (S + kQ - 1) / kQ;
    const int total = num_qt * BH;
    // Persistent: work items (query tile, (sequence, head)) are numbered longest
    // first across all heads, item i = (tile num_qt-1 - i/BH, head i%BH), and
    // dealt to the CTAs round by round in snake order (even rounds c, odd rounds
    // G-1-c), which keeps the sum of item lengths per CTA even.  Every role walks
    // the same sequence; ring slots and barrier phases follow a running key-tile
    // counter g across items.
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    struct Item {
        int qt, j0, n, b, h, g;
    };
    // Key tiles j0..qt: j0 = 0, or with a sliding window the tile holding the
    // window start of the query tile's first row (earlier tiles are never loaded).
    auto item_of = [&](int rnd, Item& it) -> bool {
        const int idx = rnd * G + ((rnd & 1) ? G - 1 - c : c);
        if (idx >= total) return false;
        it.qt = num_qt - 1 - idx / BH;
        const int ws0 = it.qt * kQ - window + 1;
        it.j0 = (kWin && ws0 > 0) ? ws0 / kKV : 0;
        it.n = it.qt + 1 - it.j0;
        const int bh = idx % BH;
        it.b = bh / H;
        it.h = bh - it.b * H;
        it.g = it.h / (H / Hkv);
        return true;
    };
    const int rounds = (total + G - 1) / G;

    if (warp == 0 && lane == 0) {
        for (int qb = 0; qb < 2; ++qb) {
            mbar_init(q_full(qb), 1);
            mbar_init(q_empty(qb), 1);
        }
        for (int s = 0; s < SK; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(k_empty(s), 1);
        }
        for (int s = 0; s < ST; ++s) {
            mbar_init(v_full(s), 1);
            mbar_init(v_empty(s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(s_full(i), 1);
            mbar_init(p_full(i), 4);
            mbar_init(o_done(i), 1);
        }
        mbar_init(done_bar, 2);              // one commit from each MMA thread
        mbar_init(l_ready, 4);               // one arrival per softmax warp
        mbar_init(o_free, 4);                // one arrival per epilogue warp
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
    // Everything above overlaps the previous kernel's tail; global memory only after.
    pdl_wait();
    pdl_trigger();
    const uint32_t t_o = tmem_base + L::kOCol;
    // Register split per warpgroup (launched with 168 per thread, 64512 in all):
    // the control warps give theirs up to the softmax, the epilogue keeps 168:
    // 128 * (80 + 232 + 168) = 61440 <= 64512.  Each warpgroup executes one
    // setmaxnreg at the top of its own branch.
    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 80;");
    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        // Per item: its Q tile once the previous item's S MMAs are done with the
        // Q buffer, then the K and V tiles in the order the MMA threads consume
        // them (K_0, then K_j, V_{j-1} for j >= 1, then V_{n-1}).  The rings run
        // on across items.  Before exiting it waits for its last load into every
        // slot, so no copy is in flight when the CTA ends.
        if (lane == 0) {
            int kn = 0, vn = 0, items = 0;           // K, V tiles and items loaded
            bool ok = true;
            Item it;
            auto load_k = [&](int j) -> bool {
                const int st = kn % SK;
                if (!mbar_wait(k_empty(st), ((uint32_t)(kn / SK) & 1u) ^ 1u, err, abort_flag)) return false;
                mbar_arrive_expect_tx(k_full(st), L::kKBytes);
#pragma unroll
                for (int sub = 0; sub < L::kSub; ++sub)
                    tma_load_3d(sK + st * L::kKBytes + sub * 16384, &kmap, 64 * sub, j * kKV,
                                it.b * Hkv + it.g, k_full(st));
                ++kn;
                return true;
            };
            auto load_v = [&](int j) -> bool {
                const int st = vn % ST;
                if (!mbar_wait(v_empty(st), ((uint32_t)(vn / ST) & 1u) ^ 1u, err, abort_flag)) return false;
                mbar_arrive_expect_tx(v_full(st), L::kVBytes);
#pragma unroll
                for (int sub = 0; sub < L::kSub; ++sub)
                    tma_load_3d(sV + st * L::kVBytes + sub * 16384, &vmap, 64 * sub, j * kKV,
                                it.b * Hkv + it.g, v_full(st));
                ++vn;
                return true;
            };
            for (int rnd = 0; rnd < rounds && ok; ++rnd) {
                if (!item_of(rnd, it)) continue;
                // Q buffer items % 2, free once item items - 2's S MMAs are done
                const int qb = items & 1;
                if (items >= 2 && !mbar_wait(q_empty(qb), (uint32_t)((items >> 1) - 1) & 1u, err, abort_flag)) break;
                mbar_arrive_expect_tx(q_full(qb), L::kQBytes);
#pragma unroll
                for (int sub = 0; sub < L::kSub; ++sub)
                    tma_load_3d(sQ + qb * L::kQBytes + sub * 16384, &qmap, 64 * sub, it.qt * kQ,
                                it.b * H + it.h, q_full(qb));
                ++items;
                ok = load_k(it.j0);
                for (int j = 1; j < it.n && ok; ++j) ok = load_k(it.j0 + j) && load_v(it.j0 + j - 1);
                if (ok) ok = load_v(it.j0 + it.n - 1);
            }
            // Drain: the copies of every armed slot (and the last Q) must land.
            for (int k = items - 2 < 0 ? 0 : items - 2; k < items; ++k)
                mbar_wait(q_full(k & 1), (uint32_t)(k >> 1) & 1u, err, abort_flag);
            for (int s = 0; s < SK && s < kn; ++s) {
                const int last = kn - 1 - ((kn - 1 - s) % SK);
                mbar_wait(k_full(s), (uint32_t)((last / SK) & 1), err, abort_flag);
            }
            for (int s = 0; s < ST && s < vn; ++s) {
                const int last = vn - 1 - ((vn - 1 - s) % ST);
                mbar_wait(v_full(s), (uint32_t)((last / ST) & 1), err, abort_flag);
            }
        }
    } else if (warp == 1 || warp == 2) {
        // ---------------------------------------------------------- MMA issuers
        // Descriptors are built once and advanced by adding (byte offset >> 4) to
        // their start-address field (shared addresses stay below 256 KB, so the
        // 14-bit field never carries).
        if (lane == 0) {
            constexpr uint32_t idesc_s = umma_idesc_bf16(kQ, kKV);
            constexpr uint32_t idesc_o = umma_idesc_bf16(kQ, DH, true);
            bool ok = true;
            int g = 0, items = 0;                    // key tiles, items so far
            Item it;
            if (warp == 1) {
                // S_g into S[g % 2] once the softmax of tile g-2 is done with it.
                const uint64_t dq = umma_desc_sw128(sQ), dk = umma_desc_sw128(sK);
                for (int rnd = 0; rnd < rounds && ok; ++rnd) {
                    if (!item_of(rnd, it)) continue;
                    const int qb = items & 1;
                    ok = mbar_wait(q_full(qb), (uint32_t)(items >> 1) & 1u, err, abort_flag);
                    const uint64_t dqi = dq + (uint64_t)((qb * L::kQBytes) >> 4);
                    for (int j = 0; j < it.n && ok; ++j, ++g) {
                        const int sb = g & 1, st = g % SK;
                        if (g >= 2 && !mbar_wait(p_full(sb), (uint32_t)((g - 2) >> 1) & 1u, err, abort_flag)) {
                            ok = false;
                            break;
                        }
                        if (!mbar_wait(k_full(st), (uint32_t)(g / SK) & 1u, err, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t d = tmem_base + (uint32_t)(sb * kKV);
                        const uint64_t kb = dk + (uint64_t)((st * L::kKBytes) >> 4);
#pragma unroll
                        for (int kk = 0; kk < DH / 16; ++kk) {
                            const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                            umma_bf16(d, dqi + off, kb + off, idesc_s, kk > 0 ? 1u : 0u);
                        }
                        umma_commit(k_empty(st));
                        umma_commit(s_full(sb));
                    }
                    // The Q buffer may be refilled once this item's S MMAs are complete.
                    if (ok) umma_commit(q_empty(qb));
                    ++items;
                }
            } else {
                // O += P_g V_g once the softmax has written P_g; the first tile of
                // an item overwrites O.
                const uint64_t dv = umma_desc_sw128_mn(sV, 16384, 1024);
                for (int rnd = 0; rnd < rounds && ok; ++rnd) {
                    if (!item_of(rnd, it)) continue;
                    // O is overwritten by this item's first P.V once the epilogue
                    // warps have read the previous item's O out of tensor memory.
                    if (items > 0 && !mbar_wait(o_free, (uint32_t)(items - 1) & 1u, err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    ++items;
                    for (int j = 0; j < it.n && ok; ++j, ++g) {
                        const int sbp = g & 1, stp = g % ST;
                        if (!mbar_wait(p_full(sbp), (uint32_t)(g >> 1) & 1u, err, abort_flag)) { ok = false; break; }
                        if (!mbar_wait(v_full(stp), (uint32_t)(g / ST) & 1u, err, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t t_p = tmem_base + L::kPCol + sbp * (kKV / 2);
                        const uint64_t vb = dv + (uint64_t)((stp * L::kVBytes) >> 4);
#pragma unroll
                        for (int kk = 0; kk < kKV / 16; ++kk)
                            umma_bf16_ts(t_o, t_p + kk * 8, vb + (uint64_t)((kk * 2048) >> 4), idesc_o,
                                         (j > 0 || kk > 0) ? 1u : 0u);
                        umma_commit(v_empty(stp));
                        umma_commit(o_done(sbp));
                    }
                }
            }
            // Every MMA this thread issued must be complete before TMEM is freed.
            umma_commit(done_bar);
            mbar_wait(done_bar, 0, err, abort_flag);
        }
    }
    } else if (warp < 8) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 232;");
        // ---------------------------------------------------------- softmax
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;                 // query row in the tile
        const uint32_t trow = tmem_base + ((uint32_t)(q4 * 32) << 16);
        const uint32_t t_orow = t_o + ((uint32_t)(q4 * 32) << 16);
        bool ok = true;
        int g = 0, items = 0;                         // key tiles, items so far
        Item it;
        for (int rnd = 0; rnd < rounds && ok; ++rnd) {
            if (!item_of(rnd, it)) continue;
            const int qt = it.qt;
            const int qi = qt * kQ + r;               // query position
            // Last visible key of this row: the diagonal, or S - 1 past the end;
            // first visible key: 0, or the window start.
            const int kmax = qi < S ? qi : S - 1;
            const int kmin = kWin ? kmax - window + 1 : 0;
            // tiles starting below this key hold keys before some row's window
            const int win_lo = kWin ? qt * kQ + kQ - window : INT_MIN;
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < it.n; ++j, ++g) {
                const int sb = g & 1;
                if (!warp_wait(s_full(sb), (uint32_t)(g >> 1) & 1u, err, abort_flag)) { ok = false; break; }
                tc_fence_after();
                // All four 32-column loads in flight before the single wait.
                uint32_t sr[kKV / 32][32];
#pragma unroll
                for (int cc = 0; cc < kKV / 32; ++cc) tmem_ld32_issue(trow + sb * kKV + cc * 32, sr[cc]);
                tmem_ld_wait();
                float s[kKV];
#pragma unroll
                for (int cc = 0; cc < kKV / 32; ++cc) {
                    reg_fence32(sr[cc]);
#pragma unroll
                    for (int e = 0; e < 32; ++e) s[cc * 32 + e] = __uint_as_float(sr[cc][e]);
                }
                const int jt = it.j0 + j;             // key tile index
                const int k0 = jt * kKV;
                // Only the diagonal tile and a tile reaching past S need the mask
                // (warp-uniform test).
                if (jt == qt || k0 + kKV > S) {
                    const int lim = kmax - k0;         // keys cc > lim are masked
#pragma unroll
                    for (int cc = 0; cc < kKV; ++cc) s[cc] = cc > lim ? -INFINITY : s[cc];
                }
                // Keys before the row's window start (CTA-uniform test); a row with
                // none left in this tile keeps m = -inf and gets p = 0 below.
                if (kWin && k0 < win_lo) {
                    const int lo = kmin - k0;          // keys cc < lo are masked
#pragma unroll
                    for (int cc = 0; cc < kKV; ++cc) s[cc] = cc < lo ? -INFINITY : s[cc];
                }
                // Row max over raw scores: four independent chains of three-input
                // maxima (the scale is positive, so it commutes with the max).
                float mx4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
                for (int cc = 4; cc < kKV; cc += 8)
#pragma unroll
                    for (int e = 0; e < 4; ++e) mx4[e] = fmax3(mx4[e], s[cc + 2 * e], s[cc + 2 * e + 1]);
                const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * scale_log2;
                float corr = 1.f;
                if (mx > m + kRescaleThreshold) {     // also true on the first tile (m = -inf)
                    corr = fast_exp2(m - mx);
                    m = mx;
                }
                const bool need_rescale = __any_sync(0xffffffffu, corr != 1.f && j > 0);
                // p = 2^(s*scale - m): scale and offset as packed pairs, one
                // exponential per element, row sum in four packed accumulators, P
                // kept in registers as bf16 pairs until its buffer is free.
                const uint64_t scale2 = f2_pack(scale_log2, scale_log2);
                // (m = -inf: no visible key yet, every p is 0)
                const float negm = (kWin && m == -INFINITY) ? 0.f : -m;
                const uint64_t negm2 = f2_pack(negm, negm);
                uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};
                uint32_t pw[kKV / 64][32];
#pragma unroll
                for (int h64 = 0; h64 < kKV / 64; ++h64) {
#pragma unroll
                    for (int e = 0; e < 64; e += 2) {
                        float t0, t1;
                        const int cc = h64 * 64 + e;
                        f2_unpack(f2_fma(f2_pack(s[cc], s[cc + 1]), scale2, negm2), t0, t1);
                        const float p0 = fast_exp2(t0), p1 = fast_exp2(t1);
                        sum2[(e >> 1) & 3] = f2_add(sum2[(e >> 1) & 3], f2_pack(p0, p1));
                        pw[h64][e >> 1] = pack_bf16x2(p0, p1);
                    }
                }
                // P[sb] is free once P_{g-2} V_{g-2} has completed; then P goes to
                // tensor memory, 64 keys (32 columns) per store.
                if (g >= 2 && !warp_wait(o_done(sb), (uint32_t)((g - 2) >> 1) & 1u, err, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t t_p = trow + L::kPCol + sb * (kKV / 2);
#pragma unroll
                for (int h64 = 0; h64 < kKV / 64; ++h64) tmem_st32_async(t_p + h64 * 32, pw[h64]);
                tmem_st_wait();
                float sa[4], sb2[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) f2_unpack(sum2[e], sa[e], sb2[e]);
                const float sum = ((sa[0] + sb2[0]) + (sa[1] + sb2[1])) + ((sa[2] + sb2[2]) + (sa[3] + sb2[3]));
                l = l * corr + sum;
                if (need_rescale) {
                    // O must hold P_{g-1} V_{g-1} before it is rescaled.
                    if (!warp_wait(o_done((g - 1) & 1), (uint32_t)((g - 1) >> 1) & 1u, err,
                                   abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int cc = 0; cc < DH / 32; ++cc) {
                        float v[32];
                        tmem_ld32(t_orow + cc * 32, v);
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] *= corr;
                        tmem_st32(t_orow + cc * 32, v);
                    }
                }
                // Before the last P of item k is published, the epilogue must have
                // taken item k-1 (its O read out, so its row-sum slot is free):
                // the softmax runs at most one item ahead of the epilogue, and
                // the wait cannot alias, since item k's O is not final before
                // this P exists.
                if (j == it.n - 1 && items > 0 &&
                    !warp_wait(o_free, (uint32_t)(items - 1) & 1u, err, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full(sb));
            }
            if (!ok) break;
            // The row sum goes to the epilogue warps, which write O / l once the
            // last P.V is done; this warp moves on to the next item.
            red_l[(items & 1) * kQ + r] = l;
            __syncwarp();
            if (lane == 0) mbar_arrive(l_ready);
            ++items;
        }
    } else {
        // ---------------------------------------------------------- epilogue
        // Per item: wait for its row sums and its last P.V, read O out of tensor
        // memory (all DH columns into registers), release O for the next item's
        // first P.V, then write O / l with heads merged, o[b, s, h*DH + d].
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;
        const uint32_t t_orow = t_o + ((uint32_t)(q4 * 32) << 16);
        int g = 0, items = 0;
        Item it;
        for (int rnd = 0; rnd < rounds; ++rnd) {
            if (!item_of(rnd, it)) continue;
            g += it.n;                                 // g - 1: this item's last key tile
            if (!warp_wait(l_ready, (uint32_t)items & 1u, err, abort_flag)) break;
            const float l = red_l[(items & 1) * kQ + r];
            if (!warp_wait(o_done((g - 1) & 1), (uint32_t)((g - 1) >> 1) & 1u, err, abort_flag)) break;
            tc_fence_after();
            uint32_t ov[DH / 32][32];
#pragma unroll
            for (int cc = 0; cc < DH / 32; ++cc) tmem_ld32_issue(t_orow + cc * 32, ov[cc]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);
            ++items;
            const int qi = it.qt * kQ + r;
            if (qi >= S) continue;
            const float inv = 1.0f / l;
            __nv_bfloat16* orow =
                o + ((int64_t)it.b * S + qi) * ((int64_t)H * DH) + (int64_t)it.h * DH;
#pragma unroll
            for (int cc = 0; cc < DH / 32; ++cc) {
                reg_fence32(ov[cc]);
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(ov[cc][e]) * inv, __uint_as_float(ov[cc][e + 1]) * inv);
                    w.y = pack_bf16x2(__uint_as_float(ov[cc][e + 2]) * inv, __uint_as_float(ov[cc][e + 3]) * inv);
                    w.z = pack_bf16x2(__uint_as_float(ov[cc][e + 4]) * inv, __uint_as_float(ov[cc][e + 5]) * inv);
                    w.w = pack_bf16x2(__uint_as_float(ov[cc][e + 6]) * inv, __uint_as_float(ov[cc][e + 7]) * inv);
                    *reinterpret_cast<uint4*>(orow + cc * 32 + e) = w;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn att_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        tried = true;
    }
    return fn;
}

// [n_seq_heads, S, dh] bf16, box min(dh, 64) x 128 x 1 with the swizzle that
// matches the box row (128 bytes: 128-byte swizzle; 64 bytes: 64-byte swizzle),
// zero fill past S.
bool heads_map(CUtensorMap* map, const void* ptr, int64_t n_seq_heads, int64_t S, int64_t dh) {
    EncodeTiledFn fn = att_encode_fn();
    if (!fn) return false;
    const cuuint32_t inner = dh >= 64 ? 64 : (cuuint32_t)dh;
    cuuint64_t dims[3] = {(cuuint64_t)dh, (cuuint64_t)S, (cuuint64_t)n_seq_heads};
    cuuint64_t strides[2] = {(cuuint64_t)(dh * 2), (cuuint64_t)(S * dh * 2)};
    cuuint32_t box[3] = {inner, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              inner * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DH, bool kWin>
cudaError_t launch_tc_w(const AttnPlan& p, cudaStream_t st) {
    using L = AttTc<DH>;
    static_assert(L::kBytes <= 232448, "shared memory budget");
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_attention_tc<DH, kWin>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    // One CTA per SM (shared memory allows no more), each looping over items.
    const int items = ((p.S + kQ - 1) / kQ) * p.B * p.H;
    const int grid = items < sm_count() ? items : sm_count();
    return launch_pdl(k_attention_tc<DH, kWin>, dim3(grid), dim3(kThreadsAtt), L::kBytes, st, p.qmap,
                      p.kmap, p.vmap, static_cast<__nv_bfloat16*>(p.o), p.B * p.H, p.H, p.Hkv,
                      p.S, p.scale * 1.4426950408889634f, p.window, device_error_word());
}

// The window is a template parameter: the full-causal instantiation keeps the
// code (and the registers) it had without the window.
template <int DH>
cudaError_t launch_tc(const AttnPlan& p, cudaStream_t st) {
    return p.window > 0 ? launch_tc_w<DH, true>(p, st) : launch_tc_w<DH, false>(p, st);
}

}  // namespace

bool attention_tc_supported(int dh) { return dh == 32 || dh == 64 || dh == 128; }

tfm_status plan_attention_tc(AttnPlan* p, const void* q, const void* k, const void* v, void* o,
                             int B, int H, int Hkv, int S, int dh, float scale) {
    p->B = B;
    p->H = H;
    p->Hkv = Hkv;
    p->S = S;
    p->dh = dh;
    p->scale = scale;
    p->o = o;
    p->window = 0;
    if (!heads_map(&p->qmap, q, (int64_t)B * H, S, dh) ||
        !heads_map(&p->kmap, k, (int64_t)B * Hkv, S, dh) ||
        !heads_map(&p->vmap, v, (int64_t)B * Hkv, S, dh))
        return TFM_ECUDA;
    return TFM_OK;
}

cudaError_t launch_attention_tc(const AttnPlan& p, cudaStream_t st) {
    if (p.B <= 0 || p.S <= 0) return cudaSuccess;
    // d_head 32: up to 256 positions, the three causal blocks of a sequence side
    // by side (k_attention_short.cu), else two query tiles per CTA as for 64;
    // d_head 64: two query tiles per CTA (k_attention_pp.cu); d_head 128: one tile
    // per CTA (two Q tiles, two P tiles and a K/V ring exceed shared memory).
    if (p.dh == 32)
        return attention_short_supported(p.dh, p.S, p.window) ? launch_attention_short(p, st)
                                                               : launch_attention_pp(p, st);
    if (p.dh == 64) return launch_attention_pp(p, st);
    if (p.dh == 128) return launch_tc<128>(p, st);
    return cudaErrorInvalidValue;
}

}  // namespace tfm
