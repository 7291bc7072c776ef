// k_gemm_skinny.cu - C[M, N] = A[M, K] . W[N, K]^T for a few rows (M <= 128),
// the projections of a decode step (one row per sequence), on the sm_103a
// tensor cores with the fused epilogues of epilogue.cuh.
//
// With M rows a GEMM is a stream of W from HBM (2 bytes per weight, 2M flops),
// bound by HBM bandwidth: what matters is that every SM keeps its share of W in
// flight.  So the operands swap roles: a 128-row slice of W is the MMA's A
// operand (M = 128) and the M rows of A, padded to NM = 16..128 rows by the
// TMA's zero fill, are its B operand (N = NM); the accumulator is a C^T tile in
// tensor memory.  K is split over the CTAs of a thread-block cluster (up to 8)
// so that tiles x splits covers the SMs:
//   warp 0      TMA producer: W box 128x64 (SwiGLU: W1 rows n..n+64 and W3 rows
//               n..n+64) and A box NMx64, 128-byte swizzle, into a ring of stages.
//               For a model weight (no launch writes it) the first stages' W
//               copies are issued before the grid dependency wait, overlapping
//               the previous kernel's tail; the A copies follow the wait.
//   warp 1      allocates the TMEM accumulator; one thread issues
//               tcgen05.mma.cta_group::1.kind::f16 (M=128, N=NM, K=16).
//   warps 2..5  read their TMEM lane quarter (one W row per thread, NM columns)
//               and store the partial C^T tile to shared memory as [NM][128] fp32.
//               With a norm input (16-row plans, GemmPlan::norm_x), they first
//               build A themselves: the RMSNorm of the residual rows (a warp per
//               row for the sums of squares, all of a row's loads in flight), then
//               each k-block's 16 x 64 bf16 tile written into its stage where the
//               TMA would have put it, their 128 arrivals joining the W copy's on
//               the stage barrier.  A decode step then needs no norm launches after
//               the first (the step measured 393.7 -> 371.0 us at the GQA workload,
//               425.7 -> 403.8 us at GPT-2-small widths, 176.9 -> 165.9 us at long
//               context: each launch removed took a kernel boundary and an L2 round
//               trip off the chain; a first form whose row sums went through
//               dependent loads, one round trip after another, was slower).
//               Their numerics are the norm kernels': r = 1 / sqrt(sum(x^2)/K + eps)
//               in fp32, then bf16(x * r * g).
// After a cluster barrier every CTA sums a share of the tile's 8-column output
// chunks over the cluster's partial tiles (distributed shared memory, split 0
// first: the result does not depend on timing) and applies the epilogue to it;
// a second cluster barrier keeps each partial tile alive until all have read it.
// Every mbarrier wait is bounded (common.cuh); on a timeout all threads still
// reach both cluster barriers.
#include "epilogue.cuh"

namespace tfm {

namespace {

constexpr int kSkThreads = 192;
constexpr int kSkBK = 64;                       // one 128-byte swizzle row of bf16
constexpr int kSkWBytes = 128 * kSkBK * 2;      // W box: 16 KB

template <int NM, int STAGES>
struct SkSmem {
    static constexpr int kXBytes = NM * kSkBK * 2;
    static constexpr int kStage = kSkWBytes + kXBytes;      // a multiple of 1024
    static constexpr int kRed = STAGES * kStage;            // partial C^T [NM][128] fp32
    static constexpr int kBar = kRed + NM * 128 * 4;        // full[S], empty[S], tfull
    static constexpr int kMisc = kBar + (2 * STAGES + 1) * 8;
    static constexpr int kBytes = kMisc + 16 + 1024;        // + alignment slack
};

// A as the RMSNorm of fp32 rows (GemmPlan::norm_x): x [M, K], gain g [K].
struct NormIn {
    const float* x;
    const float* g;
    float eps;
};

__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

template <int NM, int STAGES, bool kDual>
__global__ void __launch_bounds__(kSkThreads, 1)
    k_gemm_skinny(const __grid_constant__ TcMaps maps, int M, int N, int K, int splits,
                  int w_static, EpiParams epi, NormIn nin, int* err) {
    using L = SkSmem<NM, STAGES>;
    constexpr int kTmemCols = NM < 32 ? 32 : NM;
    constexpr int kOut = kDual ? 64 : 128;       // output columns of a tile
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t red = base + L::kRed;
    const uint32_t bars = base + L::kBar;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
    const uint32_t tfull_bar = bars + 8u * (2 * STAGES);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(gbase + L::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::kMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = (int)cluster_ctarank();    // the cluster spans the splits of one tile
    const int tile = (int)blockIdx.x / splits;
    const int n0 = tile * kOut;                  // first output column (W row) of the tile
    const int num_kb = (K + kSkBK - 1) / kSkBK;
    const int kb0 = (int)((int64_t)split * num_kb / splits);
    const int kb1 = (int)((int64_t)(split + 1) * num_kb / splits);
    const int nkb = kb1 - kb0;                   // >= 1: splits <= num_kb
    // A computed here from norm rows (16-row plans only): each stage's A tile is
    // written by warps 2..5, whose 128 arrivals join the producer's on its barrier.
    const bool fused = NM == 16 && nin.x != nullptr;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), fused ? 1 + 128 : 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(tfull_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&maps.a);
        tma_prefetch_desc(&maps.b);
        if (kDual) tma_prefetch_desc(&maps.b2);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            auto load_w = [&](int i) {
                const int s = i % STAGES;
                const uint32_t sw = base + s * L::kStage;
                const int kx = (kb0 + i) * kSkBK;
                if (kDual) {
                    tma_load_2d(sw, &maps.b, kx, n0, full_bar(s));
                    tma_load_2d(sw + 64 * kSkBK * 2, &maps.b2, kx, n0, full_bar(s));
                } else {
                    tma_load_2d(sw, &maps.b, kx, n0, full_bar(s));
                }
            };
            auto load_x = [&](int i) {
                const int s = i % STAGES;
                tma_load_2d(base + s * L::kStage + kSkWBytes, &maps.a, (kb0 + i) * kSkBK, 0,
                            full_bar(s));
            };
            const int pre = nkb < STAGES ? nkb : STAGES;
            const uint32_t tx = fused ? (uint32_t)kSkWBytes : (uint32_t)L::kStage;
            if (!w_static) pdl_wait();           // W may come from the launch before
            for (int i = 0; i < pre; ++i) {
                mbar_arrive_expect_tx(full_bar(i), tx);
                load_w(i);
            }
            pdl_wait();
            pdl_trigger();
            if (!fused)
                for (int i = 0; i < pre; ++i) load_x(i);
            for (int i = pre; i < nkb; ++i) {
                const int s = i % STAGES;
                if (!mbar_wait(empty_bar(s), (uint32_t)(((i / STAGES) - 1) & 1), err, abort_flag))
                    break;
                mbar_arrive_expect_tx(full_bar(s), tx);
                load_w(i);
                if (!fused) load_x(i);
            }
        } else {
            pdl_wait();
            pdl_trigger();
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        pdl_wait();
        pdl_trigger();
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_bf16(128, NM);
            for (int i = 0; i < nkb; ++i) {
                const int s = i % STAGES;
                if (!mbar_wait(full_bar(s), (uint32_t)((i / STAGES) & 1), err, abort_flag)) break;
                tc_fence_after();
                const uint32_t sw = base + s * L::kStage;
                const uint32_t sx = sw + kSkWBytes;
#pragma unroll
                for (int k = 0; k < kSkBK / 16; ++k)
                    umma_bf16(tmem_base, umma_desc_sw128(sw + k * 32), umma_desc_sw128(sx + k * 32),
                              idesc, (i > 0 || k > 0) ? 1u : 0u);
                umma_commit(empty_bar(s));
            }
            umma_commit(tfull_bar);
        }
    } else {
        // ---------------------------------------------------------- TMEM -> shared
        pdl_wait();
        pdl_trigger();
        const int q = warp & 3;                  // TMEM lane quarter of this warp
        bool conv_ok = true;
        if (fused) {
            // ------------------------------------------------ A from the norm rows
            // The RMSNorm of the CS336 walkthrough (section 5.6) with the same
            // arithmetic as the norm kernels: r = 1 / sqrt(sum(x^2) / K + eps) in
            // fp32, then bf16(x * r * g).  For the tiles thread ct owns row ct / 8,
            // 16-byte chunk ct % 8 (8 columns) of each k-block's 16 x 64 tile, stored
            // where a 128-byte-swizzled TMA box would put it (chunk j of row r at
            // j ^ r % 8).
            const int ct = (int)threadIdx.x - 64;
            const int row = ct >> 3, ch = ct & 7;
            const float* xrow = nin.x + (int64_t)(row < M ? row : 0) * K;
            // Prefetch ring over the k-blocks, one slot per stage; the first
            // stages' loads are issued before the sums, so the two overlap.
            float4 xa[STAGES][2], ga[STAGES][2];
            auto fetch = [&](int i, int u) {
                const int kx = (kb0 + i) * kSkBK + ch * 8;
                const bool in = i < nkb && row < M && kx < K;
                const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                xa[u][0] = in ? __ldg(reinterpret_cast<const float4*>(xrow + kx)) : z;
                xa[u][1] = in ? __ldg(reinterpret_cast<const float4*>(xrow + kx + 4)) : z;
                ga[u][0] = in ? __ldg(reinterpret_cast<const float4*>(nin.g + kx)) : z;
                ga[u][1] = in ? __ldg(reinterpret_cast<const float4*>(nin.g + kx + 4)) : z;
            };
#pragma unroll
            for (int u = 0; u < STAGES; ++u) fetch(u, u);
            // Sums of squares: warp w takes rows w, w + 4, ...; lane l the float4
            // groups l, l + 32, ... of the row, sixteen loads in flight at a time,
            // then a shuffle reduction (the summation order of the norm kernels).
            float* red = reinterpret_cast<float*>(gbase + L::kRed);   // [16], free until the MMAs end
            const int k4 = K >> 2;
            for (int m = warp - 2; m < M; m += 4) {
                const float4* xr = reinterpret_cast<const float4*>(nin.x + (int64_t)m * K);
                float ssum = 0.f;
                for (int c0 = 0; c0 < k4; c0 += 32 * 16) {
                    float4 v[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const int c = c0 + lane + 32 * u;
                        v[u] = c < k4 ? __ldg(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        ssum += v[u].x * v[u].x + v[u].y * v[u].y + v[u].z * v[u].z + v[u].w * v[u].w;
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
                if (lane == 0) red[m] = ssum;
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");   // warps 2..5 only
            float rinv = 0.f;                                // rows >= M are zero
            if (row < M) rinv = 1.0f / sqrtf(red[row] / (float)K + nin.eps);
            for (int i0 = 0; i0 < nkb && conv_ok; i0 += STAGES) {
#pragma unroll
                for (int u = 0; u < STAGES; ++u) {
                    const int i = i0 + u;                    // stage u
                    if (i >= nkb) break;
                    if (i >= STAGES &&
                        !warp_wait(empty_bar(u), (uint32_t)(((i / STAGES) - 1) & 1), err, abort_flag)) {
                        conv_ok = false;
                        break;
                    }
                    const float4 a0 = xa[u][0], a1 = xa[u][1], g0 = ga[u][0], g1 = ga[u][1];
                    const uint32_t sx = base + (uint32_t)(u * L::kStage + kSkWBytes);
                    st_shared_v4(sx + row * 128 + ((ch ^ (row & 7)) << 4),
                                 pack_bf16x2(a0.x * rinv * g0.x, a0.y * rinv * g0.y),
                                 pack_bf16x2(a0.z * rinv * g0.z, a0.w * rinv * g0.w),
                                 pack_bf16x2(a1.x * rinv * g1.x, a1.y * rinv * g1.y),
                                 pack_bf16x2(a1.z * rinv * g1.z, a1.w * rinv * g1.w));
                    fence_proxy_async_smem();           // read by the tensor cores
                    mbar_arrive(full_bar(u));
                    fetch(i + STAGES, u);
                }
            }
        }
        if (conv_ok && warp_wait(tfull_bar, 0, err, abort_flag)) {
            tc_fence_after();
            const int r = q * 32 + lane;         // W row of the tile held by this thread
            float* part = reinterpret_cast<float*>(gbase + L::kRed);
#pragma unroll
            for (int c = 0; c < (NM + 31) / 32; ++c) {
                uint32_t v[32];
                tmem_ld32_issue(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 32), v);
                tmem_ld_wait();
                // All 32 destinations stay live until the wait: the load writes
                // them asynchronously, so a register the compiler saw as dead
                // (columns past NM) must not be handed to another value meanwhile.
                reg_fence32(v);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (c * 32 + j < NM && c * 32 + j < M) part[(c * 32 + j) * 128 + r] = __uint_as_float(v[j]);
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync();                              // every partial tile of the cluster is stored
    tc_fence_after();
    // This CTA's share of the tile's output chunks: 8 columns of one row each.
    constexpr int kChunksPerRow = kOut / 8;
    const int nchunk = M * kChunksPerRow;
    for (int ci = split * kSkThreads + (int)threadIdx.x; ci < nchunk; ci += splits * kSkThreads) {
        const int m = ci / kChunksPerRow, j0 = (ci - m * kChunksPerRow) * 8;
        float a[8], u[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] = u[e] = 0.f;
        for (int s = 0; s < splits; ++s) {
            const uint32_t src = mapa_shared(red + (uint32_t)((m * 128 + j0) * 4), (uint32_t)s);
            const float4 x0 = ld_dsmem_f4(src), x1 = ld_dsmem_f4(src + 16);
            a[0] += x0.x; a[1] += x0.y; a[2] += x0.z; a[3] += x0.w;
            a[4] += x1.x; a[5] += x1.y; a[6] += x1.z; a[7] += x1.w;
            if (kDual) {                          // the up rows sit 64 rows below the gate rows
                const float4 y0 = ld_dsmem_f4(src + 256), y1 = ld_dsmem_f4(src + 272);
                u[0] += y0.x; u[1] += y0.y; u[2] += y0.z; u[3] += y0.w;
                u[4] += y1.x; u[5] += y1.y; u[6] += y1.z; u[7] += y1.w;
            }
        }
        apply_epilogue<8>(epi, m, n0 + j0, a, u);
    }
    cluster_sync();                              // no CTA leaves while its tile may be read
    if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

template <int NM, int STAGES, bool kDual>
cudaError_t skinny_inst(const GemmPlan& p, cudaStream_t st) {
    using L = SkSmem<NM, STAGES>;
    static_assert(L::kBytes <= 232448, "shared memory budget");
    static bool attr_set = false;   // per instantiation; set once per process
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm_skinny<NM, STAGES, kDual>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.sk_tiles * p.sk_splits));
    cfg.blockDim = dim3(kSkThreads);
    cfg.dynamicSmemBytes = L::kBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)p.sk_splits;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const NormIn nin{p.norm_x, p.norm_g, p.norm_eps};
    return cudaLaunchKernelEx(&cfg, k_gemm_skinny<NM, STAGES, kDual>, p.maps, p.M, p.N, p.K,
                              p.sk_splits, p.b_static, p.epi, nin, device_error_word());
}

// Ring depth per NM: the W stages of two CTAs per SM (NM <= 32) or of one.
template <bool kDual>
cudaError_t skinny_dispatch(const GemmPlan& p, cudaStream_t st) {
    switch (p.sk_nm) {
        case 16: return skinny_inst<16, 5, kDual>(p, st);
        case 32: return skinny_inst<32, 4, kDual>(p, st);
        case 64: return skinny_inst<64, 6, kDual>(p, st);
        case 128: return skinny_inst<128, 4, kDual>(p, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_gemm_skinny(const GemmPlan& p, cudaStream_t st) {
    return p.dual ? skinny_dispatch<true>(p, st) : skinny_dispatch<false>(p, st);
}

}  // namespace tfm
