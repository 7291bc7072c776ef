// k_attention_pp.cu - causal softmax attention on tcgen05, two query tiles per
// CTA whose softmax phases alternate ("ping-pong"), for d_head 32 and 64 (the
// library uses it for 64).
//
// Same mathematics as k_attention_tc.cu (CS336 walkthrough, section 5.4;
// "LLM 2", section GQA / MQA): o = softmax(q k^T / sqrt(dh) + M) v, online over
// key tiles of 128 with a lazily rescaled running max.  What differs is the
// schedule.  A work item is the pair of query tiles A = 2p and B = 2p + 1 of one
// (sequence, head), and every key/value tile is loaded once for both.  The
// kernel is persistent: one CTA per SM walks a list of items (longest first
// across all heads, dealt in snake order), with Q double-buffered so the next
// item's loads overlap the current one's tail:
//   warp 0      TMA: Q_A and Q_B of each item, then K_j and V_j into two rings
//   warp 1      TMEM (S_A, S_B: 128 columns each; O_A, O_B: dh each; P_A, P_B:
//               64 each) and the S MMAs: S_x = Q_x K_j^T for x = A, B
//   warp 10     the P.V MMAs: O_x += P_x V_j, P_x read from tensor memory
//   warps 2..5  softmax of tile A, warps 6..9 softmax of tile B (one thread per
//               query row), so while one group runs its exponentials the other's
//               scores are being computed and the two groups share the issue slots
//               and the special-function unit of each scheduler.
// The softmax works on packed fp32 pairs (f32x2 FMA/ADD) and three-input
// maxima, about 3 instructions per score besides the exponential (the
// special-function unit takes 4 cycles per warp ex2 on each scheduler; the
// bf16 packing and the FMAs overlap with it).  (Evaluating part of the
// exponentials with a polynomial on the FMA pipe was measured slower here: it
// costs more issue slots than it frees.  Taking an unmasked tile's row maximum
// from the tensor-memory load with tcgen05.ld.red measured faster, 144.7 ->
// 134.1 us at long context.  It is not used, because with it one
// prefill-against-forward bit-equality check failed: a 37-position sequence
// whose only key tile is masked, so that path never uses the hardware maximum.
// The likely cause: on that path the load's maximum outputs were dead while the
// asynchronous load could still write them, so their registers may have been
// reused meanwhile.  Every destination of an asynchronous load has to stay live
// until its wait.)  S_x(j+1) is issued as soon as the
// softmax of tile x has read S_x(j) into registers, P_x.V_j as soon as it has
// written P_x(j); the exponentials of tile j+1 run before the wait for P_x.V_j
// (which frees the P_x columns), so that wait overlaps them.  (Two threads per
// row, 16 softmax warps exchanging partial row maxima through shared memory,
// was measured slower: the bounded barrier round trip of the exchange costs
// ~600 cycles per tile and the two tiles fall into lockstep.  So was a separate
// epilogue warpgroup writing O out, as the d_head 128 kernel does, at 16 warps
// with a setmaxnreg split: long 139 -> 164 us, gpt2s 28 -> 33 us.)  An MMA warp
// shares its scheduler with two softmax warps, which leaves it few issue slots;
// one thread issuing all ~24 MMAs of a key tile was measured to be the bound,
// hence two issuing threads.  Making the two warps of a lane quarter (one per
// tile, same scheduler) take turns at the exponentials, as a strict A, B, A, ...
// alternation through a pair of barriers per quarter, was measured slower
// (long attention 154 -> 170 us, whole launch): one warp alone runs the
// exponentials at ~6 cycles per ex2, two in step at ~4.3, the special-function
// unit's rate.  The packed forms ex2.approx.ftz.bf16x2 and ex2.approx.f16x2 take
// 8 cycles per warp instruction, the same 32 results per cycle per SM as the f32
// form, so packing P's exponentials gains nothing.  Splitting the tile into four
// 32-column chunks, each loaded from tensor memory while the previous one runs
// its exponentials against the running maximum (raised, with the earlier chunks'
// P rescaled, when a chunk passes it by the threshold), was correct but much
// slower (long 140.5 -> 191 us, gpt2s 28.8 -> 38.5 us): S_x can be released only
// after its last chunk is loaded, which holds back the next S MMA that each
// tile's softmax then waits for.  All waits are bounded; tiles above the
// diagonal are never loaded.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace tfm {

namespace {

constexpr int kQ = 128;
constexpr int kKV = 128;
constexpr int kThreadsPP = 352;
constexpr float kRescaleThresholdPP = 8.0f;   // log2 units: P entries stay below 2^8

template <int DH>
struct AttPP {
    static constexpr int kRowBytes = DH * 2;                 // 64 (dh 32) or 128 (dh 64)
    static constexpr int kStages = DH == 64 ? 5 : 6;
    static constexpr int kQBytes = kQ * DH * 2;
    static constexpr int kKBytes = kKV * DH * 2;
    static constexpr int kVBytes = kKV * DH * 2;
    static constexpr int kQOff = 0;                          // two buffers of Q_A, Q_B
    static constexpr int kKOff = kQOff + 4 * kQBytes;
    static constexpr int kVOff = kKOff + kStages * kKBytes;
    static constexpr int kBarOff = kVOff + kStages * kVBytes;
    // Tensor-memory columns: S_A, S_B (128 each), O_A, O_B (DH each), then P_A,
    // P_B (64 each: 128 bf16 per row, two per 32-bit column).
    static constexpr int kOCol = 2 * kKV;
    static constexpr int kPCol = kOCol + 2 * DH;
    // q_full[0], k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2], p_full[2],
    // o_done[2], done, s_free[2], q_empty[2], q_full[1]
    static constexpr int kNumBars = 1 + 4 * kStages + 12;
    static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
    static constexpr int kBytes = kMiscOff + 16 + 1024;
    // Shared-memory descriptor swizzle of the Q/K/V tiles: 128-byte rows use the
    // 128-byte swizzle (code 2), 64-byte rows the 64-byte swizzle (code 4).
    static constexpr uint32_t kSwz = DH == 32 ? 4u : 2u;
    static constexpr uint32_t kGroup = 8 * kRowBytes;        // 8-row swizzle atom
};

template <int DH, bool kWin>
__global__ void __launch_bounds__(kThreadsPP, 1)
    k_attention_pp(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, __nv_bfloat16* __restrict__ o, int BH,
                   int H, int Hkv, int S, float scale_log2, int window, int* err) {
    using L = AttPP<DH>;
    constexpr int ST = L::kStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t sQ = base + L::kQOff, sK = base + L::kKOff, sV = base + L::kVOff;
    const uint32_t bars = base + L::kBarOff;
    // Q is double-buffered: item k uses buffer k % 2.
    auto q_full = [&](int qb) { return qb == 0 ? bars : bars + 8u * (12 + 4 * ST); };
    auto q_empty = [&](int qb) { return bars + 8u * (10 + 4 * ST + qb); };
    auto k_full = [&](int s) { return bars + 8u * (1 + s); };
    auto k_empty = [&](int s) { return bars + 8u * (1 + ST + s); };
    auto v_full = [&](int s) { return bars + 8u * (1 + 2 * ST + s); };
    auto v_empty = [&](int s) { return bars + 8u * (1 + 3 * ST + s); };
    auto s_full = [&](int x) { return bars + 8u * (1 + 4 * ST + x); };
    auto p_full = [&](int x) { return bars + 8u * (3 + 4 * ST + x); };
    auto o_done = [&](int x) { return bars + 8u * (5 + 4 * ST + x); };
    const uint32_t done_bar = bars + 8u * (7 + 4 * ST);
    auto s_free = [&](int x) { return bars + 8u * (8 + 4 * ST + x); };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(gbase + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_qt = (S + kQ - 1) / kQ;
    const int num_pairs = (num_qt + 1) / 2;
    const int total = num_pairs * BH;
    // Persistent: work items (pair p of (sequence, head) bh) are numbered longest
    // first across all heads, item i = (pair num_pairs-1 - i/BH, head i%BH), and
    // dealt to the CTAs round by round in snake order (even rounds c, odd rounds
    // G-1-c), which keeps the sum of item lengths per CTA even.  Every role walks
    // the same sequence; barrier phases follow running counters across items.
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    // Key tiles j0 + j for j in [0, nmax): j0 = 0, or with a sliding window the
    // tile holding tile A's first window start (earlier tiles are never loaded);
    // query tile x uses j in [lo[x], n[x]).
    struct Item {
        int qA, qB, j0, lo[2], n[2], nmax, b, h, g;
    };
    auto item_of = [&](int rnd, Item& it) -> bool {
        const int idx = rnd * G + ((rnd & 1) ? G - 1 - c : c);
        if (idx >= total) return false;
        const int pair = num_pairs - 1 - idx / BH;
        const int bh = idx % BH;
        it.b = bh / H;
        it.h = bh - it.b * H;
        it.g = it.h / (H / Hkv);
        it.qA = 2 * pair;
        it.qB = 2 * pair + 1;
        const int wsA = it.qA * kQ - window + 1, wsB = it.qB * kQ - window + 1;
        const int jA = (kWin && wsA > 0) ? wsA / kKV : 0;
        const int jB = (kWin && wsB > 0) ? wsB / kKV : 0;
        it.j0 = jA;
        it.lo[0] = 0;
        it.n[0] = it.qA + 1 - jA;                                // key tiles of tile A
        it.lo[1] = it.qB < num_qt ? jB - jA : 0;
        it.n[1] = it.qB < num_qt ? it.qB + 1 - jA : 0;           // 0: tile B does not exist
        it.nmax = it.n[1] > it.n[0] ? it.n[1] : it.n[0];
        return true;
    };
    const int rounds = (total + G - 1) / G;

    if (warp == 0 && lane == 0) {
        for (int qb = 0; qb < 2; ++qb) {
            mbar_init(q_full(qb), 1);
            mbar_init(q_empty(qb), 1);
        }
        for (int s = 0; s < ST; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(k_empty(s), 1);
            mbar_init(v_full(s), 1);
            mbar_init(v_empty(s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(s_full(x), 1);
            mbar_init(p_full(x), 4);
            mbar_init(o_done(x), 1);
            mbar_init(s_free(x), 4);
        }
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

    constexpr uint32_t idesc_s = umma_idesc_bf16(kQ, kKV);
    constexpr uint32_t idesc_o = umma_idesc_bf16(kQ, DH, true);
    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        // Per item k: Q_A and Q_B into Q buffer k % 2 (once item k-2's S MMAs are
        // done with it), then K_j and V_j into the two rings, which run on across
        // items, so the next item's loads overlap this item's tail.  Before exiting
        // it waits for its last load into every slot, so no copy is in flight when
        // the CTA ends.
        if (lane == 0) {
            int kv = 0, items = 0;
            bool ok = true;
            Item it;
            for (int rnd = 0; rnd < rounds && ok; ++rnd) {
                if (!item_of(rnd, it)) continue;
                const int qb = items & 1;
                if (items >= 2 &&
                    !mbar_wait(q_empty(qb), (uint32_t)((items >> 1) - 1) & 1u, err, abort_flag))
                    break;
                const uint32_t sq = sQ + qb * 2 * L::kQBytes;
                mbar_arrive_expect_tx(q_full(qb), 2 * L::kQBytes);
                tma_load_3d(sq, &qmap, 0, it.qA * kQ, it.b * H + it.h, q_full(qb));
                tma_load_3d(sq + L::kQBytes, &qmap, 0, it.qB * kQ, it.b * H + it.h, q_full(qb));
                ++items;
                for (int j = 0; j < it.nmax; ++j) {
                    const int st = kv % ST;
                    const uint32_t ph = ((uint32_t)(kv / ST) & 1u) ^ 1u;
                    if (!mbar_wait(k_empty(st), ph, err, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(k_full(st), L::kKBytes);
                    tma_load_3d(sK + st * L::kKBytes, &kmap, 0, (it.j0 + j) * kKV, it.b * Hkv + it.g,
                                k_full(st));
                    if (!mbar_wait(v_empty(st), ph, err, abort_flag)) {
                        mbar_wait(k_full(st), (uint32_t)((kv / ST) & 1), err, abort_flag);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(v_full(st), L::kVBytes);
                    tma_load_3d(sV + st * L::kVBytes, &vmap, 0, (it.j0 + j) * kKV, it.b * Hkv + it.g,
                                v_full(st));
                    ++kv;
                }
            }
            for (int k = items - 2 < 0 ? 0 : items - 2; k < items; ++k)
                mbar_wait(q_full(k & 1), (uint32_t)(k >> 1) & 1u, err, abort_flag);
            for (int s = 0; s < ST && s < kv; ++s) {
                const int last = kv - 1 - ((kv - 1 - s) % ST);
                mbar_wait(k_full(s), (uint32_t)((last / ST) & 1), err, abort_flag);
                mbar_wait(v_full(s), (uint32_t)((last / ST) & 1), err, abort_flag);
            }
        }
    } else if (warp == 1 || warp == 10) {
        // ---------------------------------------------------------- MMA issuers
        // Two threads on different schedulers: warp 1 issues S_x = Q_x K_j^T (into
        // the S columns), warp 10 issues O_x += P_x V_j (P from its TMEM columns).
        // The two streams touch disjoint tensor memory and are ordered only through
        // the softmax barriers; each commit covers its own thread's MMAs.  Both
        // share the scheduler with two busy softmax warps, so the per-MMA work is
        // kept small: descriptors are built once and advanced by adding
        // (byte offset >> 4) to their start-address field (shared addresses stay
        // below 256 KB, so the 14-bit field never carries).
        if (lane == 0) {
            bool ok = true;
            int kv = 0, items = 0, cnt[2] = {0, 0};   // K/V tiles, items, MMAs per tile x
            Item it;
            if (warp == 1) {
                const uint64_t dq = sdesc(sQ, L::kSwz, 16, L::kGroup);
                const uint64_t dk = sdesc(sK, L::kSwz, 16, L::kGroup);
                auto issue_s = [&](int qb, int x, int st) {
                    const uint64_t a0 = dq + (uint64_t)((qb * 2 + x) * (L::kQBytes >> 4));
                    const uint64_t b0 = dk + (uint64_t)(st * (L::kKBytes >> 4));
                    const uint32_t t_s = tmem_base + x * kKV;
#pragma unroll
                    for (int kk = 0; kk < DH / 16; ++kk)
                        umma_bf16(t_s, a0 + 2 * kk, b0 + 2 * kk, idesc_s, kk > 0 ? 1u : 0u);
                    umma_commit(s_full(x));
                };
                for (int rnd = 0; rnd < rounds && ok; ++rnd) {
                    if (!item_of(rnd, it)) continue;
                    const int qb = items & 1;
                    ok = mbar_wait(q_full(qb), (uint32_t)(items >> 1) & 1u, err, abort_flag);
                    for (int j = 0; j < it.nmax && ok; ++j) {
                        const int st = kv % ST;
                        ok = mbar_wait(k_full(st), (uint32_t)(kv / ST) & 1u, err, abort_flag);
                        for (int x = 0; x < 2 && ok; ++x) {
                            if (j < it.lo[x] || j >= it.n[x]) continue;
                            // S_x is free once the softmax has read the previous
                            // scores into registers (possibly of the previous item).
                            if (cnt[x] > 0)
                                ok = mbar_wait(s_free(x), (uint32_t)(cnt[x] - 1) & 1u, err, abort_flag);
                            if (ok) {
                                tc_fence_after();
                                issue_s(qb, x, st);
                                ++cnt[x];
                            }
                        }
                        if (ok) umma_commit(k_empty(st));
                        ++kv;
                    }
                    // Q buffer qb may be refilled once this item's S MMAs are complete.
                    if (ok) umma_commit(q_empty(qb));
                    ++items;
                }
            } else {
                const uint64_t dv = sdesc(sV, L::kSwz, 0, L::kGroup);
                auto issue_pv = [&](int x, int st, bool first) {
                    const uint64_t b0 = dv + (uint64_t)(st * (L::kVBytes >> 4));
                    const uint32_t t_o = tmem_base + L::kOCol + x * DH;
                    const uint32_t t_p = tmem_base + L::kPCol + x * (kKV / 2);
#pragma unroll
                    for (int kk = 0; kk < kKV / 16; ++kk)
                        umma_bf16_ts(t_o, t_p + kk * 8, b0 + kk * ((16 * L::kRowBytes) >> 4),
                                     idesc_o, (!first || kk > 0) ? 1u : 0u);
                    umma_commit(o_done(x));
                };
                for (int rnd = 0; rnd < rounds && ok; ++rnd) {
                    if (!item_of(rnd, it)) continue;
                    for (int j = 0; j < it.nmax && ok; ++j) {
                        const int st = kv % ST;
                        ok = mbar_wait(v_full(st), (uint32_t)(kv / ST) & 1u, err, abort_flag);
                        for (int x = 0; x < 2 && ok; ++x) {
                            if (j < it.lo[x] || j >= it.n[x]) continue;
                            // The first P of an item is written only after the
                            // softmax has read the previous item's O_x, so the
                            // overwrite (first = true) cannot race that read.
                            ok = mbar_wait(p_full(x), (uint32_t)cnt[x] & 1u, err, abort_flag);
                            if (ok) {
                                tc_fence_after();
                                issue_pv(x, st, j == it.lo[x]);
                                ++cnt[x];
                            }
                        }
                        if (ok) umma_commit(v_empty(st));
                        ++kv;
                    }
                }
            }
            // Every MMA this thread issued must be complete before TMEM is freed
            // (done_bar counts one commit from each issuer).
            umma_commit(done_bar);
            mbar_wait(done_bar, 0, err, abort_flag);
        }
    } else {
        // ---------------------------------------------------------- softmax (warps 2..9)
        const int x = (warp - 2) >> 2;                 // 0: tile A, 1: tile B
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const uint32_t t_s = tmem_base + x * kKV + lane_off;
        const uint32_t t_o = tmem_base + L::kOCol + x * DH + lane_off;
        const uint32_t t_p = tmem_base + L::kPCol + x * (kKV / 2) + lane_off;
        int cnt = 0;                                   // tiles of this x processed so far
        bool ok = true;
        Item it;
        for (int rnd = 0; rnd < rounds && ok; ++rnd) {
            if (!item_of(rnd, it)) continue;
            const int n = it.n[x];
            if (n == 0) continue;
            const int qt = x == 0 ? it.qA : it.qB;
            const int qi = qt * kQ + r;
            // first visible key: 0, or the window start of the row (rows past S
            // take the window of row S - 1)
            const int kmin = kWin ? (qi < S ? qi : S - 1) - window + 1 : 0;
            const int win_lo = kWin ? qt * kQ + kQ - window : INT_MIN;
            float m = -INFINITY, l = 0.f;
            for (int j = it.lo[x]; j < n && ok; ++j, ++cnt) {
                if (!warp_wait(s_full(x), (uint32_t)cnt & 1u, err, abort_flag)) { ok = false; break; }
                tc_fence_after();
                uint32_t sr[kKV / 32][32];
#pragma unroll
                for (int cc = 0; cc < kKV / 32; ++cc) tmem_ld32_issue(t_s + cc * 32, sr[cc]);
                tmem_ld_wait();
                // S_x is in registers: the tensor cores may overwrite it with the next tile.
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_free(x));
                float s[kKV];
#pragma unroll
                for (int cc = 0; cc < kKV / 32; ++cc) {
                    reg_fence32(sr[cc]);
#pragma unroll
                    for (int e = 0; e < 32; ++e) s[cc * 32 + e] = __uint_as_float(sr[cc][e]);
                }
                const int jt = it.j0 + j;              // key tile index
                const int k0 = jt * kKV;
                if (jt == qt || k0 + kKV > S) {
#pragma unroll
                    for (int cc = 0; cc < kKV; ++cc)
                        if (k0 + cc > qi || k0 + cc >= S) s[cc] = -INFINITY;
                }
                // Keys before the row's window start (CTA-uniform test); a row with
                // none left in this tile keeps m = -inf and gets p = 0 below.
                if (kWin && k0 < win_lo) {
#pragma unroll
                    for (int cc = 0; cc < kKV; ++cc)
                        if (k0 + cc < kmin) s[cc] = -INFINITY;
                }
                // Row max: four independent chains of three-input maxima.
                float mx4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
                for (int cc = 4; cc < kKV; cc += 8)
#pragma unroll
                    for (int e = 0; e < 4; ++e) mx4[e] = fmax3(mx4[e], s[cc + 2 * e], s[cc + 2 * e + 1]);
                const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * scale_log2;
                float corr = 1.f;
                if (mx > m + kRescaleThresholdPP) {
                    corr = fast_exp2(m - mx);
                    m = mx;
                }
                const bool need_rescale = __any_sync(0xffffffffu, corr != 1.f && j > it.lo[x]);
                // p = 2^(s*scale - m): scale and offset as packed pairs, one exponential
                // per element, row sum in four packed accumulators, P kept in registers
                // as bf16 pairs.  The exponentials do not depend on the previous P.V,
                // so they run before the wait for it.
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
                // P_x and O_x are free once the previous O_x += P_x V (possibly of the
                // previous item) has completed; then P goes to tensor memory, 64 keys
                // (32 columns) per store.
                if (cnt > 0 && !warp_wait(o_done(x), (uint32_t)(cnt - 1) & 1u, err, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int h64 = 0; h64 < kKV / 64; ++h64) tmem_st32_async(t_p + h64 * 32, pw[h64]);
                tmem_st_wait();
                float sa[4], sb[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) f2_unpack(sum2[e], sa[e], sb[e]);
                const float sum = ((sa[0] + sb[0]) + (sa[1] + sb[1])) + ((sa[2] + sb[2]) + (sa[3] + sb[3]));
                l = l * corr + sum;
                if (need_rescale) {
                    tc_fence_after();
#pragma unroll
                    for (int cc = 0; cc < DH / 32; ++cc) {
                        float v[32];
                        tmem_ld32(t_o + cc * 32, v);
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] *= corr;
                        tmem_st32(t_o + cc * 32, v);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full(x));
            }
            // O_x of this item is complete after its last P.V; read it out before
            // the next item's first P is published (its P.V overwrites O_x).
            if (ok && warp_wait(o_done(x), (uint32_t)(cnt - 1) & 1u, err, abort_flag)) {
                tc_fence_after();
                const float inv = 1.0f / l;
                __nv_bfloat16* orow =
                    o + ((int64_t)it.b * S + qi) * ((int64_t)H * DH) + (int64_t)it.h * DH;
#pragma unroll
                for (int cc = 0; cc < DH / 32; ++cc) {
                    float v[32];
                    tmem_ld32(t_o + cc * 32, v);
                    if (qi < S) {
#pragma unroll
                        for (int e = 0; e < 32; e += 8) {
                            uint4 w;
                            w.x = pack_bf16x2(v[e] * inv, v[e + 1] * inv);
                            w.y = pack_bf16x2(v[e + 2] * inv, v[e + 3] * inv);
                            w.z = pack_bf16x2(v[e + 4] * inv, v[e + 5] * inv);
                            w.w = pack_bf16x2(v[e + 6] * inv, v[e + 7] * inv);
                            *reinterpret_cast<uint4*>(orow + cc * 32 + e) = w;
                        }
                    }
                }
            } else {
                ok = false;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

template <int DH, bool kWin>
cudaError_t launch_pp_w(const AttnPlan& p, cudaStream_t st) {
    using L = AttPP<DH>;
    static_assert(L::kBytes <= 232448, "shared memory budget");
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_attention_pp<DH, kWin>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    // One CTA per SM (shared memory allows no more), each looping over items.
    const int num_qt = (p.S + kQ - 1) / kQ;
    const int items = ((num_qt + 1) / 2) * p.B * p.H;
    const int grid = items < sm_count() ? items : sm_count();
    return launch_pdl(k_attention_pp<DH, kWin>, dim3(grid), dim3(kThreadsPP), L::kBytes, st, p.qmap,
                      p.kmap, p.vmap, static_cast<__nv_bfloat16*>(p.o), p.B * p.H, p.H, p.Hkv,
                      p.S, p.scale * 1.4426950408889634f, p.window, device_error_word());
}

// The window is a template parameter: the full-causal instantiation keeps the
// code (and the registers) it had without the window.
template <int DH>
cudaError_t launch_pp(const AttnPlan& p, cudaStream_t st) {
    return p.window > 0 ? launch_pp_w<DH, true>(p, st) : launch_pp_w<DH, false>(p, st);
}

}  // namespace

cudaError_t launch_attention_pp(const AttnPlan& p, cudaStream_t st) {
    if (p.B <= 0 || p.S <= 0) return cudaSuccess;
    if (p.dh == 32) return launch_pp<32>(p, st);
    if (p.dh == 64) return launch_pp<64>(p, st);
    return cudaErrorInvalidValue;
}

}  // namespace tfm
