// k_gemm_tc.cu - bf16 GEMM on the sm_103a tensor cores with fused epilogues.
//
// C[M, N] = A[M, K] . B[N, K]^T with both operands K-major (row-major, K
// contiguous): the bias-free Linear of the CS336 walkthrough (section 5.3,
// y = x W^T with W stored (out_features, in_features)).  fp32 accumulation in
// tensor memory; the epilogue (epilogue.cuh) applies the fused residual add,
// silu*mul, or RoPE + head split.
//
// Structure (one CTA per SM, persistent over 128 x BN output tiles):
//   warp 0      TMA producer: A box 128x64 and B box BNx64 (bf16, 128-byte
//               swizzle) into a STAGES-deep shared-memory ring (full/empty mbarriers)
//   warp 1      allocates 2*BN TMEM columns; one thread issues
//               tcgen05.mma.cta_group::1.kind::f16 (M=128, N=BN, K=16) into one of two
//               TMEM accumulators, tcgen05.commit frees ring slots and hands the
//               finished accumulator to the epilogue
//   warps 2..9  epilogue, two warps per TMEM lane quarter (warp w reads lanes
//               32*(w%4).., the pair takes alternate 32-column chunks): tcgen05.ld,
//               compute the fused output (one row per thread), transpose the 32x32
//               block through swizzled shared memory and write it with coalesced
//               16-byte stores (row segments of whole sectors), or with 16-byte fp32
//               reductions at L2 for the residual add.  A warp can keep only a few
//               stores in flight, so the store rate scales with the number of
//               storing warps; measured, a 32x32 chunk costs ~700-1000 cycles per warp.
// Double-buffered accumulators let the epilogue of tile i overlap the MMAs of
// tile i+1.  For SwiGLU (kDual) a B tile is [W1 rows n..n+BN/2; W3 rows
// n..n+BN/2] so matching gate and up columns land in the same tile without
// repacking the weights.  Every mbarrier wait is bounded (common.cuh).
#include "epilogue.cuh"

#include <mutex>

namespace tfm {

constexpr int kBM = 128;                 // tile rows = UMMA M
constexpr int kBK = 64;                  // one 128-byte swizzle row of bf16
constexpr int kUmmaK = 16;               // K per tcgen05.mma kind::f16
constexpr int kTileABytes = kBM * kBK * 2;
constexpr int kEpiWarps = 8;             // two per TMEM lane quarter
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kStageOutBytes = 32 * 128; // one 32 x 32 block (fp32 rows of 128 B) per warp

// kPair: a CTA pair shares one 256 x BN tile; each CTA holds 128 rows of A and
// BN/2 rows of B per stage.
template <int BN, int STAGES, bool kPair = false>
struct TcSmem {
    static constexpr int kTileBBytes = (kPair ? BN / 2 : BN) * kBK * 2;
    static constexpr int kStageBytes = kTileABytes + kTileBBytes;
    static constexpr int kOutOffset = STAGES * kStageBytes;              // epilogue staging
    static constexpr int kBarOffset = kOutOffset + kEpiWarps * kStageOutBytes;
    // full[S], empty[S], tfull[2], tempty[2], done
    static constexpr int kNumBars = 2 * STAGES + 5;
    static constexpr int kMiscOffset = kBarOffset + kNumBars * 8;
    static constexpr int kBytes = kMiscOffset + 16 + 1024;   // + alignment slack
};


// Thread `lane` writes row `lane` of a 32 x 32 block into the staging buffer:
// fp32 rows of 128 bytes (16-byte chunk j of row r at position j ^ (r % 8)) or
// bf16 rows of 64 bytes (chunk j at j ^ ((r / 2) % 4)).  The XOR keeps both
// this row-wise write and the segment-wise read below free of bank conflicts.
__device__ __forceinline__ void stage_row(uint32_t buf, int lane, const float (&o)[32], bool bf16) {
    if (bf16) {
        const uint32_t row = buf + lane * 64;
        const int x = (lane >> 1) & 3;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            st_shared_v4(row + ((j ^ x) << 4), pack_bf16x2(o[8 * j], o[8 * j + 1]),
                         pack_bf16x2(o[8 * j + 2], o[8 * j + 3]),
                         pack_bf16x2(o[8 * j + 4], o[8 * j + 5]),
                         pack_bf16x2(o[8 * j + 6], o[8 * j + 7]));
    } else {
        const uint32_t row = buf + lane * 128;
        const int x = lane & 7;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            st_shared_v4(row + ((j ^ x) << 4), __float_as_uint(o[4 * j]),
                         __float_as_uint(o[4 * j + 1]), __float_as_uint(o[4 * j + 2]),
                         __float_as_uint(o[4 * j + 3]));
    }
}

// Writes the staged 32 x 32 block (rows row0.., columns col..) to its
// destination with each lane moving one 16-byte row segment per step, so a warp
// store covers whole 32-byte sectors.  Rows >= M and columns >= N are skipped
// exactly (element-wise at a ragged right edge).  All shared-memory reads of
// the block are issued before the first global store: the reads are ordered
// against memory operations, so interleaving them would serialise the steps.
__device__ __forceinline__ void flush_block(const EpiParams& p, uint32_t buf, int lane, int row0,
                                            int col) {
    if (p.kind == EPI_STORE_F32 || p.kind == EPI_ACCUM_F32) {
        const int seg = lane & 7;
        const int ncol = col + seg * 4;
        uint4 vs[8];
#pragma unroll
        for (int step = 0; step < 8; ++step) {
            const int r = step * 4 + (lane >> 3);
            vs[step] = ld_shared_v4(buf + r * 128 + ((seg ^ (r & 7)) << 4));
        }
#pragma unroll
        for (int step = 0; step < 8; ++step) {
            const int r = step * 4 + (lane >> 3);
            const uint4 v = vs[step];
            const int row = row0 + r;
            if (row >= p.M || ncol >= p.N) continue;
            float* d = static_cast<float*>(p.out) + (int64_t)row * p.ldo + ncol;
            if (ncol + 4 <= p.N) {
                if (p.kind == EPI_STORE_F32)
                    *reinterpret_cast<uint4*>(d) = v;
                else
                    red_add_v4_f32(d, v);
            } else {
                const float f[4] = {__uint_as_float(v.x), __uint_as_float(v.y),
                                    __uint_as_float(v.z), __uint_as_float(v.w)};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (ncol + e < p.N) {
                        if (p.kind == EPI_STORE_F32) d[e] = f[e];
                        else atomicAdd(d + e, f[e]);
                    }
            }
        }
        return;
    }
    // bf16 destinations: 4 lanes per 64-byte row, 8 rows per step.
    const int seg = lane & 3;
    QkvSlot qs{};
    __nv_bfloat16* qbase = nullptr;
    if (p.kind == EPI_QKV_ROPE) {
        qs = qkv_slot(p, col);
        qbase = static_cast<__nv_bfloat16*>(qs.region == 0 ? p.q : (qs.region == 1 ? p.k : p.v));
    }
    const int ncol = col + seg * 8;
    uint4 vs[4];
#pragma unroll
    for (int step = 0; step < 4; ++step) {
        const int r = step * 8 + (lane >> 2);
        vs[step] = ld_shared_v4(buf + r * 64 + ((seg ^ ((r >> 1) & 3)) << 4));
    }
    // QKV: (batch, position) of this lane's first row, advanced by 8 rows a step
    int qb = 0, qpos = 0;
    if (p.kind == EPI_QKV_ROPE) {
        const int row = row0 + (lane >> 2);
        qb = row / p.S;
        qpos = row - qb * p.S;
    }
#pragma unroll
    for (int step = 0; step < 4; ++step) {
        const int r = step * 8 + (lane >> 2);
        const uint4 v = vs[step];
        const int row = row0 + r;
        const int b = qb, pos = qpos;
        if (p.kind == EPI_QKV_ROPE) {
            qpos += 8;
            while (qpos >= p.S) { qpos -= p.S; ++qb; }
        }
        if (row >= p.M || ncol >= p.N) continue;
        __nv_bfloat16* d;
        if (p.kind == EPI_QKV_ROPE) {
            d = qbase + qkv_offset(p, qs, b, pos) + seg * 8;
        } else {
            d = static_cast<__nv_bfloat16*>(p.out) + (int64_t)row * p.ldo + ncol;
        }
        if (ncol + 8 <= p.N) {
            *reinterpret_cast<uint4*>(d) = v;
        } else {
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (ncol + e < p.N)
                    d[e] = __ushort_as_bfloat16((unsigned short)((w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu));
        }
    }
}

// Writes the staged 32 x 32 block (rows row0.., columns col..) with one TMA
// store (a reduce-add for the residual kind) issued by the calling thread; the
// tensor map clips rows >= M and columns >= N.  The staging layouts are the
// maps' swizzles: fp32 rows of 128 bytes (128-byte swizzle), bf16 rows of 64
// bytes (64-byte swizzle).  QKV blocks lie inside one sequence (S % 32 == 0)
// and one head (dh % 32 == 0): (d0, s0, b*heads + head) in its [B*heads, S, dh]
// map.
__device__ __forceinline__ void tma_out_block(const TcMaps& maps, const EpiParams& p, uint32_t buf,
                                              int row0, int col) {
    if (row0 >= p.M || col >= p.N) return;
    switch (p.kind) {
        case EPI_ACCUM_F32:
            tma_reduce_add_2d(&maps.out, buf, col, row0);
            break;
        case EPI_QKV_ROPE: {
            const QkvSlot q = qkv_slot(p, col);
            const int b = row0 / p.S;
            const CUtensorMap* m = q.region == 0 ? &maps.oq : (q.region == 1 ? &maps.ok : &maps.ov);
            tma_store_3d(m, buf, q.d0, row0 - b * p.S, b * q.heads + q.head);
            break;
        }
        default:
            tma_store_2d(&maps.out, buf, col, row0);
            break;
    }
}

// kExt: the epilogues of the second model family and the fused loss (a bias
// vector, EPI_LSE); without it those paths are compiled out, so the plans that
// need neither keep the code they had without them.
template <int BN, int STAGES, bool kDual, bool kPair, bool kExt>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_tc(const __grid_constant__ TcMaps maps, int M, int N, int K, int n_fast, EpiParams epi,
              int* err) {
    using L = TcSmem<BN, STAGES, kPair>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const uint32_t sA0 = base;
    const uint32_t sB0 = base + STAGES * kTileABytes;
    const uint32_t sOut = base + L::kOutOffset;
    const uint32_t bars = base + L::kBarOffset;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bars + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bars + 8u * (2 * STAGES + 2 + a); };
    const uint32_t done_bar = bars + 8u * (2 * STAGES + 4);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(gbase + L::kMiscOffset);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::kMiscOffset + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_per_tile = kDual ? BN / 2 : BN;
    // A pair's tile has 256 rows: rank 0 holds rows [0, 128), rank 1 [128, 256).
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;
    const int tile_rows = kPair ? 2 * kBM : kBM;
    const int num_m = (M + tile_rows - 1) / tile_rows;
    const int num_n = (N + n_per_tile - 1) / n_per_tile;
    const int num_tiles = num_m * num_n;
    const int num_kb = (K + kBK - 1) / kBK;
    const int unit = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;   // tile scheduler slot
    const int units = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    const bool leader = rank == 0;
    // Tile t -> (row block, column block): column blocks fastest when A is the
    // larger operand (the tiles in flight then share a few A row blocks and read
    // all of B, which stays in L2), row blocks fastest otherwise.
    auto tile_m = [&](int t) { return n_fast ? t / num_n : t % num_m; };
    auto tile_n = [&](int t) { return n_fast ? t % num_n : t / num_m; };

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), kPair ? 2 * kEpiWarps : kEpiWarps);   // both CTAs' epilogues
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&maps.a);
        tma_prefetch_desc(&maps.b);
        if (kDual) tma_prefetch_desc(&maps.b2);
    }
    if (warp == 1) {
        if (kPair) tmem_alloc_pair(smem_u32(tmem_holder), 2 * BN);
        else tmem_alloc(smem_u32(tmem_holder), 2 * BN);
    }
    tc_fence_before();
    // The pair's barriers must be initialised before either CTA signals the other's.
    if (kPair) cluster_sync();
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // Everything above overlaps the previous kernel's tail; global memory only after.
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int t = unit; t < num_tiles && ok; t += units) {
                const int m0 = tile_m(t) * tile_rows + (int)rank * kBM;
                const int n0 = tile_n(t) * n_per_tile;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, err, abort_flag)) { ok = false; break; }
                    const uint32_t sa = sA0 + stage * kTileABytes;
                    const uint32_t sb = sB0 + stage * L::kTileBBytes;
                    if (kPair) {
                        // Both CTAs' copies complete on the leader's full barrier; the
                        // leader announces the bytes of both.
                        const uint32_t fb = mapa_shared(full_bar(stage), 0);
                        if (leader) mbar_arrive_expect_tx(full_bar(stage), 2 * L::kStageBytes);
                        tma_load_2d_pair(sa, &maps.a, kb * kBK, m0, fb);
                        if (kDual)   // rank 0: W1 rows, rank 1: W3 rows of the same columns
                            tma_load_2d_pair(sb, leader ? &maps.b : &maps.b2, kb * kBK, n0, fb);
                        else
                            tma_load_2d_pair(sb, &maps.b, kb * kBK, n0 + (int)rank * (BN / 2), fb);
                    } else {
                        mbar_arrive_expect_tx(full_bar(stage), L::kStageBytes);
                        tma_load_2d(sa, &maps.a, kb * kBK, m0, full_bar(stage));
                        if (kDual) {
                            tma_load_2d(sb, &maps.b, kb * kBK, n0, full_bar(stage));
                            tma_load_2d(sb + (BN / 2) * kBK * 2, &maps.b2, kb * kBK, n0, full_bar(stage));
                        } else {
                            tma_load_2d(sb, &maps.b, kb * kBK, n0, full_bar(stage));
                        }
                    }
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // Drain: every armed stage's last phase must have landed before exit.  In
            // a pair only the leader's full barriers exist; they count the peer's
            // copies too, and the closing cluster barrier holds the peer until then.
            for (int s = 0; s < STAGES && issued > 0 && leader; ++s) {
                if (s >= issued) break;
                const int64_t last = issued - 1 - ((issued - 1 - s) % STAGES);
                mbar_wait(full_bar(s), (uint32_t)((last / STAGES) & 1), err, abort_flag);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        // In a pair only the leader issues: M = 256 over both CTAs' operands;
        // the commits arrive on the barriers of both CTAs.
        if (lane == 0 && leader) {
            constexpr uint32_t idesc = umma_idesc_bf16(kPair ? 2 * kBM : kBM, BN);
            constexpr uint16_t kBoth = 3;
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = unit; t < num_tiles && ok; t += units) {
                if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, err, abort_flag)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(full_bar(stage), phase, err, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = sA0 + stage * kTileABytes;
                    const uint32_t sb = sB0 + stage * L::kTileBBytes;
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        const uint64_t ad = umma_desc_sw128(sa + k * kUmmaK * 2);
                        const uint64_t bd = umma_desc_sw128(sb + k * kUmmaK * 2);
                        if (kPair) umma_bf16_pair(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                        else umma_bf16(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    if (kPair) umma_commit_pair(empty_bar(stage), kBoth);
                    else umma_commit(empty_bar(stage));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (kPair) umma_commit_pair(tfull_bar(acc), kBoth);
                else umma_commit(tfull_bar(acc));
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            // All MMAs this thread issued must be complete before TMEM is freed.
            if (kPair) umma_commit_pair(done_bar, 1);
            else umma_commit(done_bar);
            mbar_wait(done_bar, 0, err, abort_flag);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;                       // TMEM lane quarter of this warp
        const int half = (warp - 2) >> 2;             // the two warps of a quarter split the chunks
        const uint32_t stg = sOut + (uint32_t)((warp - 2) * kStageOutBytes);
        const bool obf = !(epi.kind == EPI_STORE_F32 || epi.kind == EPI_ACCUM_F32);
        // QKV with d_head <= 64: every chunk this warp takes starts at the same
        // offset inside its head (chunks step by 64 columns), so the thread's
        // (cos, sin) pairs are the same for all of them.  They are loaded once per
        // tile, before the accumulator wait, instead of once per chunk.
        const bool rope_pre = epi.kind == EPI_QKV_ROPE && epi.dh <= 64 && epi.rope_cs && !epi.bias;
        const int rope_d0 = (half * 32) % epi.dh;
        const int rot_cols = (epi.n_head + epi.n_kv_head) * epi.dh;   // q and k columns
        float rcs[32];
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t nblk = 0;                            // blocks written by TMA (buffer parity)
        // Rank 1 releases the accumulator on the leader's barrier.
        const uint32_t tempty0 = kPair ? mapa_shared(tempty_bar(0), 0) : tempty_bar(0);
        for (int t = unit; t < num_tiles; t += units) {
            const int m0 = tile_m(t) * tile_rows + (int)rank * kBM;
            const int n0 = tile_n(t) * n_per_tile;
            if (rope_pre) {
                const int r = m0 + q * 32 + lane;
                const int pos = epi_pos0(epi) + (r < M ? r : 0) % epi.S;
                load_vec<32>(epi.rope_cs + ((int64_t)pos * (epi.dh / 2) + rope_d0 / 2) * 2, rcs);
            }
            if (!warp_wait(tfull_bar(acc), acc_phase, err, abort_flag)) break;
            tc_fence_after();
            const int row0 = m0 + q * 32;
            const int row = row0 + lane;
            const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            // Chunks of 32 columns in range; the warp-uniform count keeps every
            // .sync.aligned TMEM load converged.
            const int left = N - n0;
            const int nck = (left >= n_per_tile ? n_per_tile : left + 31) / 32;

            auto process = [&](const uint32_t (&ra)[32], const uint32_t (&ru)[32], int c) {
                const int col = n0 + c * 32;
                float a[32], u[32], o[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    a[e] = __uint_as_float(ra[e]);
                    u[e] = __uint_as_float(ru[e]);
                }
                if (rope_pre) {
                    if (col < rot_cols) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float x0 = a[2 * j], x1 = a[2 * j + 1];
                            o[2 * j] = x0 * rcs[2 * j] - x1 * rcs[2 * j + 1];
                            o[2 * j + 1] = x0 * rcs[2 * j + 1] + x1 * rcs[2 * j];
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = a[j];
                    }
                } else {
                    epi_compute<32, kExt>(epi, row, col, a, u, o);
                }
                if (epi.tma_out && col + 32 <= N) {
                    // One bulk copy per block, issued by lane 0; a bf16 block (2 KB)
                    // alternates between the halves of the warp's 4 KB buffer, an fp32
                    // block fills it.  A buffer is rewritten once the copy issued from
                    // it has read it.  (Only blocks whole in N: a tensor store was seen
                    // to write the rest of the last 16-byte segment past N, so a
                    // ragged right edge takes the per-lane stores, which stop exactly.)
                    const uint32_t buf = stg + (obf ? (nblk & 1u) * 2048u : 0u);
                    if (lane == 0) {
                        if (obf) bulk_wait_read<1>();
                        else bulk_wait_read<0>();
                    }
                    __syncwarp();
                    stage_row(buf, lane, o, obf);
                    fence_proxy_async_smem();         // the block is read by the async proxy
                    __syncwarp();
                    if (lane == 0) {
                        tma_out_block(maps, epi, buf, row0, col);
                        bulk_commit();
                    }
                    ++nblk;
                } else {
                    if (epi.tma_out) {                // no bulk copy may still read the buffer
                        if (lane == 0) bulk_wait_read<0>();
                        __syncwarp();
                    }
                    stage_row(stg, lane, o, obf);
                    __syncwarp();
                    flush_block(epi, stg, lane, row0, col);
                    __syncwarp();                     // the buffer is reused by the next chunk
                }
            };
            // This warp takes every other chunk; a TMEM load costs only a few tens
            // of cycles, the global stores dominate, so more storing warps (not
            // deeper load pipelining) is what raises the epilogue's throughput.
            if (kExt && epi.kind == EPI_LSE) {
                // Fused cross-entropy: nothing is stored but, per row, the running
                // max and sum of exp(z - max) over this warp's chunks of the tile,
                // and the logit of the target column where the tile holds it.
                constexpr float kLog2e = 1.4426950408889634f;
                const int trg = row < M ? __ldg(epi.targets + row) : -1;
                float mx = -INFINITY, sm = 0.f, tv = 0.f;
                bool has_t = false;
#pragma unroll 1
                for (int c = half; c < nck; c += 2) {
                    uint32_t ra[32];
                    __syncwarp();
                    tmem_ld32_issue(trow + c * 32, ra);
                    tmem_ld_wait();
                    reg_fence32(ra);
                    const int col = n0 + c * 32;
                    if (epi.bias) {                      // a biased LM head
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (col + e < N)
                                ra[e] = __float_as_uint(__uint_as_float(ra[e]) + __ldg(epi.bias + col + e));
                    }
                    float cm = -INFINITY;
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (col + e < N) cm = fmaxf(cm, __uint_as_float(ra[e]));
                    const float nm = fmaxf(mx, cm);      // finite: the chunk has a column < N
                    float acc = 0.f;
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (col + e < N) acc += exp2f((__uint_as_float(ra[e]) - nm) * kLog2e);
                    sm = sm * exp2f((mx - nm) * kLog2e) + acc;   // 2^-inf = 0 on the first chunk
                    mx = nm;
                    if (trg >= col && trg < col + 32) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (col + e == trg) tv = __uint_as_float(ra[e]);
                        has_t = true;
                    }
                }
                if (row < M) {
                    epi.lse_part[(int64_t)row * epi.lse_slots + tile_n(t) * 2 + half] =
                        make_float2(mx, sm);
                    if (has_t) epi.lse_tgt[row] = tv;
                }
            } else {
#pragma unroll 1
                for (int c = half; c < nck; c += 2) {
                    uint32_t ra[32], ru[32];
                    __syncwarp();
                    tmem_ld32_issue(trow + c * 32, ra);
                    if (kDual) tmem_ld32_issue(trow + BN / 2 + c * 32, ru);
                    tmem_ld_wait();
                    reg_fence32(ra);
                    if (kDual) reg_fence32(ru);
                    process(ra, kDual ? ru : ra, c);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (kPair) mbar_arrive_cluster(tempty0 + 8u * acc);
                else mbar_arrive(tempty_bar(acc));
            }
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        // Every bulk copy this warp issued has completed before the CTA ends.
        if (epi.tma_out && lane == 0) bulk_wait<0>();
    }

    tc_fence_before();
    // A pair frees its tensor memory together and neither CTA leaves while the
    // other may still read its shared memory.
    if (kPair) cluster_sync();
    else __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        if (kPair) tmem_dealloc_pair(tmem_base, 2 * BN);
        else tmem_dealloc(tmem_base, 2 * BN);
    }
}

// ------------------------------------------------------------------ host side
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// bf16 operand [rows, cols] (row stride ld), box box_rows x 64, 128-byte swizzle,
// zero fill out of range.
bool make_operand_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld,
                      int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tile width minimising (waves x tile width), the per-SM critical path when
// every tile costs time proportional to its width.  A 128-wide tile moves 25%
// more operand bytes from L2 per flop than a 256-wide one (85 vs 64 flop per
// byte), so its cost carries a 1.25 factor; ties go to the wider tile.
int choose_block_n(int M, int N, bool dual) {
    const int sms = sm_count();
    const int num_m = (M + kBM - 1) / kBM;
    int best = 256;
    double best_cost = -1.0;
    for (int bn : {256, 128}) {
        const int per = dual ? bn / 2 : bn;
        const int64_t tiles = (int64_t)num_m * ((N + per - 1) / per);
        // A 128-wide tile was measured to take ~0.8 of a 256-wide one (the same
        // A tile, fill and MMA issue per tile), so it wins only by saving a wave.
        const double cost = (double)((tiles + sms - 1) / sms) * bn * (bn == 128 ? 1.6 : 1.0);
        if (best_cost < 0 || cost < best_cost) { best = bn; best_cost = cost; }
    }
    return best;
}

template <int BN, int STAGES, bool kDual, bool kPair = false, bool kExt = false>
cudaError_t launch_inst(const GemmPlan& p, cudaStream_t st) {
    using L = TcSmem<BN, STAGES, kPair>;
    static_assert(L::kBytes <= 232448, "shared memory budget");
    static bool attr_set = false;   // per instantiation; set once per process
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm_tc<BN, STAGES, kDual, kPair, kExt>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int per = kDual ? BN / 2 : BN;
    const int rows = kPair ? 2 * kBM : kBM;
    const int64_t tiles = (int64_t)((p.M + rows - 1) / rows) * ((p.N + per - 1) / per);
    const int slots = kPair ? sm_count() / 2 : sm_count();
    const int units = (int)(tiles < slots ? tiles : slots);
    if (kPair)
        return launch_pdl_pair(k_gemm_tc<BN, STAGES, kDual, kPair, kExt>, dim3(2 * units), dim3(kThreads),
                               L::kBytes, st, p.maps, p.M, p.N, p.K, p.n_fast, p.epi,
                               device_error_word());
    return launch_pdl(k_gemm_tc<BN, STAGES, kDual, kPair, kExt>, dim3(units), dim3(kThreads), L::kBytes,
                      st, p.maps, p.M, p.N, p.K, p.n_fast, p.epi, device_error_word());
}

}  // namespace

// Output map for the epilogue's TMA stores: [rows, cols] fp32 (128-byte swizzle)
// or bf16 (64-byte swizzle), row stride ld elements, box 32 x 32.
bool make_out_map(CUtensorMap* map, void* ptr, int64_t rows, int64_t cols, int64_t ld, bool bf16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int es = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * es)};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr,
              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              bf16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Head-major bf16 output [n_seq_heads, S, dh], box 32 (of dh) x 32 (positions) x 1.
bool make_heads_out_map(CUtensorMap* map, void* ptr, int64_t n_seq_heads, int64_t S, int64_t dh) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)dh, (cuuint64_t)S, (cuuint64_t)n_seq_heads};
    cuuint64_t strides[2] = {(cuuint64_t)(dh * 2), (cuuint64_t)(S * dh * 2)};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16_ptr(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The epilogue writes through TMA when the destination allows it: 16-byte
// aligned base and row stride; QKV only when no 32-row block crosses a sequence
// (S % 32 == 0) and blocks tile the heads (dh % 32 == 0).  Otherwise it keeps
// the per-lane stores.  Plain fp32 stores (the LM head's logits) keep them too:
// a 4 KB fp32 block fills a warp's staging buffer, so each block waited for the
// previous one's bulk read, and the LM head was measured slower (gpt2s 539 ->
// 576 us) where the bf16 QKV blocks, two per buffer, were faster (gpt2s 32.5 ->
// 28.8 us) and the fp32 reduce-add about even.
bool plan_tma_out(TcMaps* maps, const EpiParams& e) {
    switch (e.kind) {
        case EPI_ACCUM_F32:
            return e.out && aligned16_ptr(e.out) && (e.ldo * 4) % 16 == 0 &&
                   make_out_map(&maps->out, e.out, e.M, e.N, e.ldo, false);
        case EPI_STORE_BF16:
            return e.out && aligned16_ptr(e.out) && (e.ldo * 2) % 16 == 0 &&
                   make_out_map(&maps->out, e.out, e.M, e.N, e.ldo, true);
        case EPI_SWIGLU:
        case EPI_GELU:
            return e.out_bf16 && e.out && aligned16_ptr(e.out) && (e.ldo * 2) % 16 == 0 &&
                   make_out_map(&maps->out, e.out, e.M, e.N, e.ldo, true);
        case EPI_QKV_ROPE: {
            if (!e.out_bf16 || e.S <= 0 || e.S % 32 != 0 || e.dh % 32 != 0 || e.M % e.S != 0 ||
                e.kv_stride != 0)
                return false;
            if (!aligned16_ptr(e.q) || !aligned16_ptr(e.k) || !aligned16_ptr(e.v)) return false;
            const int64_t B = e.M / e.S;
            return make_heads_out_map(&maps->oq, e.q, B * e.n_head, e.S, e.dh) &&
                   make_heads_out_map(&maps->ok, e.k, B * e.n_kv_head, e.S, e.dh) &&
                   make_heads_out_map(&maps->ov, e.v, B * e.n_kv_head, e.S, e.dh);
        }
        default:
            return false;
    }
}

tfm_status plan_gemm_tc(GemmPlan* plan, const void* A, int64_t lda, const void* B, const void* B2,
                        int64_t ldb, int M, int N, int K, const EpiParams& epi) {
    const bool dual = B2 != nullptr;
    plan->M = M;
    plan->N = N;
    plan->K = K;
    plan->dual = dual ? 1 : 0;
    plan->skinny = 0;
    plan->b_static = 0;
    plan->norm_x = nullptr;
    plan->norm_g = nullptr;
    plan->norm_eps = 0.f;
    if (M <= kBM && epi.kind != EPI_LSE) {
        // A few rows: stream W over all SMs (k_gemm_skinny.cu).  Tiles of 128 W
        // rows (64 output columns for SwiGLU); K split so that tiles x splits
        // fills the SMs, two CTAs per SM where a CTA's ring fits twice.
        plan->skinny = 1;
        plan->pair = 0;
        plan->n_fast = 0;
        plan->block_n = 128;
        plan->sk_nm = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
        const int out = dual ? 64 : 128;
        plan->sk_tiles = (N + out - 1) / out;
        const int num_kb = (K + kBK - 1) / kBK;
        const int slots = sm_count() * (plan->sk_nm <= 32 ? 2 : 1);
        int splits = slots / plan->sk_tiles;
        if (splits > 8) splits = 8;              // portable cluster size
        if (splits > num_kb) splits = num_kb;
        plan->sk_splits = splits < 1 ? 1 : splits;
        plan->epi = epi;
        plan->epi.tma_out = 0;
        if (!make_operand_map(&plan->maps.a, A, M, K, lda, plan->sk_nm)) return TFM_ECUDA;
        if (!make_operand_map(&plan->maps.b, B, N, K, ldb, dual ? 64 : 128)) return TFM_ECUDA;
        if (dual) {
            if (!make_operand_map(&plan->maps.b2, B2, N, K, ldb, 64)) return TFM_ECUDA;
        } else {
            plan->maps.b2 = plan->maps.b;
        }
        return TFM_OK;
    }
    // CTA pairs (256 x 256 tiles, half of B per SM): per k-block each SM holds
    // 32 KB instead of 48 KB, so six stages are in flight and a long main loop
    // keeps up with the tensor cores.  With a short K the tile time is set by the
    // epilogue's stores, and the pair (whose accumulator is released only when
    // both CTAs' epilogues are done) was measured slower; so pairs are used for
    // K >= 2048, or K >= 1024 with N >= 2048 or many waves of tiles.  (At
    // K = 1024: long-context QKV, N = 3072, 46.1 -> 43.1 us with pairs; the
    // output projection, N = 1024, unchanged; pairs for every K >= 1024 made the
    // short workload's down projection, N = 512, K = 1344, slower: 18.9 -> 20.3 us.)
    {
        const int64_t pair_tiles = (int64_t)((M + 2 * kBM - 1) / (2 * kBM)) *
                                   ((N + (dual ? 127 : 255)) / (dual ? 128 : 256));
        const bool long_k = K >= 2048 ||
                            (K >= 1024 && (N >= 2048 || pair_tiles >= 8LL * (sm_count() / 2)));
        plan->pair = (M > kBM && long_k) ? 1 : 0;
    }
    plan->block_n = plan->pair ? 256 : choose_block_n(M, N, dual);
    // Column blocks fastest when A (M x K bf16) is larger than B and too large
    // to stay in L2 (over 64 MB): with row blocks fastest every wave streams all
    // of A once per column block, and at gqa the down projection (A 92 MB, B
    // 23 MB) read 444 MB from DRAM against 182 MB algorithmic (194 MB in the
    // other order, 124 -> 118 us).  Where A fits in L2 the order was measured
    // neutral to slower (QKV gqa 75 -> 79 us), so it stays row blocks fastest.
    const int64_t a_bytes = (int64_t)M * K * 2, b_bytes = (int64_t)N * (dual ? 2 : 1) * K * 2;
    plan->n_fast = (a_bytes > b_bytes && a_bytes > (64ll << 20)) ? 1 : 0;
    plan->epi = epi;
    const int box_b = (dual || plan->pair) ? plan->block_n / 2 : plan->block_n;
    if (!make_operand_map(&plan->maps.a, A, M, K, lda, kBM)) return TFM_ECUDA;
    if (!make_operand_map(&plan->maps.b, B, N, K, ldb, box_b)) return TFM_ECUDA;
    if (dual) {
        if (!make_operand_map(&plan->maps.b2, B2, N, K, ldb, box_b)) return TFM_ECUDA;
    } else {
        plan->maps.b2 = plan->maps.b;
    }
    plan->epi.tma_out = plan_tma_out(&plan->maps, plan->epi) ? 1 : 0;
    return TFM_OK;
}

template <bool kExt>
cudaError_t launch_gemm_tc_ext(const GemmPlan& p, cudaStream_t st) {
    if (p.pair) {
        if (p.dual) return launch_inst<256, 6, true, true, kExt>(p, st);
        return launch_inst<256, 6, false, true, kExt>(p, st);
    }
    if (p.dual) {
        if (p.block_n == 256) return launch_inst<256, 4, true, false, kExt>(p, st);
        return launch_inst<128, 6, true, false, kExt>(p, st);
    }
    if (p.block_n == 256) return launch_inst<256, 4, false, false, kExt>(p, st);
    return launch_inst<128, 6, false, false, kExt>(p, st);
}

cudaError_t launch_gemm_tc(const GemmPlan& p, cudaStream_t st) {
    if (p.M <= 0 || p.N <= 0) return cudaSuccess;
    if (p.skinny) return launch_gemm_skinny(p, st);
    if (p.epi.bias || p.epi.kind == EPI_LSE) return launch_gemm_tc_ext<true>(p, st);
    return launch_gemm_tc_ext<false>(p, st);
}

}  // namespace tfm
