// router.cu -- the routing components of WIDE (Sec. 3.1 "Routing
// Components", Eq. 4-5, inference branch) on tcgen05:
//
//   z[t, j]    = sum_d X[t,d] W1[j,d]            (bottleneck, j < r)
//   R[t, g, c] = sum_j z[t,j] W2[2g+c, j]        (2 N_G outputs reshaped to (N_G, 2))
//   mask[t, g] = 1 when argmax_c R[t,g,c] = 0, i.e. R[t,g,0] >= R[t,g,1]
//
// The router reads X once and is bound by HBM (2 r flop per X byte).  A
// persistent CTA owns 128 token rows: TMA streams X tiles (the M = 128 side)
// and W1 tiles (the N = r side) into a pipeline as deep as shared memory
// allows next to W2 (up to 10 stages), one thread issues tcgen05.mma with
// the fp32 accumulator in TMEM (double-buffered across tiles), and sixteen
// epilogue warps (eight for r = 64) -- four (two) per TMEM lane quadrant, one
// token row per thread, each taking a share of the groups -- read z from TMEM, form the logits with
// fp32 FMAs in ascending j against W2 held in shared memory (four groups at
// a time, eight independent chains), and write the mask row (and optionally
// the logits).
//
// route_reorder (REORDER = true) adds the mask reordering (Eq. 7) to the same
// launch.  The epilogue warps also ballot every group's decisions over their
// 32 token rows and store the four ballots of each (tile, group) in the
// workspace; after a grid barrier each CTA scans one group's per-tile active
// counts into tile offsets and counts[g]; after a second barrier each CTA
// places the tokens of its own tiles: active token at offset + rank among the
// tile's active tokens, inactive token after counts[g] likewise -- the stable
// partition, bit for bit.  The launch is cooperative (every CTA resident), and
// the barriers are bounded waits on a counter in the workspace.
#include "common.cuh"
#include "internal.h"
#include "partition.cuh"

namespace wide {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
// warp 0 TMA, warp 1 MMA + TMEM, then the epilogue warps: four per TMEM lane
// quadrant for r <= 32, two for r = 64 (whose z row needs twice the registers)
template <int R> __host__ __device__ constexpr int epi_warps() { return R >= 64 ? 8 : 16; }
template <int R> __host__ __device__ constexpr int router_threads() { return 32 * (2 + epi_warps<R>()); }
constexpr int kMaxStages = 10;
constexpr int kW2MaxBytes = 64 * 1024;
constexpr int kSmemBudget = 225 * 1024;

template <int R>
struct RouterCfg {
    static_assert(R == 16 || R == 32 || R == 64, "router bottleneck width");
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = R * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * R < 32 ? 32 : 2 * R;
    static constexpr uint32_t IDESC = idesc_bf16_f32(BM, R);
    static constexpr int BAR_BYTES = 256;
    static_assert(STAGE_BYTES % 1024 == 0, "SW128 operand alignment");
    static_assert((2 * kMaxStages + 5) * 8 + 8 <= BAR_BYTES, "barrier area");
    static_assert(1024 + 2 * STAGE_BYTES + kW2MaxBytes + BAR_BYTES <= kSmemBudget, "two stages fit");
    // stages next to a W2 of w2_bytes, and the dynamic shared memory that takes
    static int stages(int w2_bytes) {
        const int n = (kSmemBudget - 1024 - BAR_BYTES - ((w2_bytes + 15) & ~15)) / STAGE_BYTES;
        return n > kMaxStages ? kMaxStages : n;
    }
    static int smem_bytes(int w2_bytes) {
        return 1024 + stages(w2_bytes) * STAGE_BYTES + ((w2_bytes + 15) & ~15) + BAR_BYTES;
    }
};

template <int R, bool REORDER>
__global__ void __launch_bounds__(router_threads<R>(), 1)
    router_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW1,
                  const RouterArgs args) {
    using C = RouterCfg<R>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int n_stages = args.stages;
    const int w2_bytes = 2 * args.n_groups * R * 2;
    uint8_t *stages = smem;
    uint16_t *w2s = reinterpret_cast<uint16_t *>(smem + n_stages * C::STAGE_BYTES);  // [2 ng][R]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + n_stages * C::STAGE_BYTES + ((w2_bytes + 15) & ~15));
    uint64_t *full = bars;
    uint64_t *empty = bars + n_stages;
    uint64_t *tfull = bars + 2 * n_stages;
    uint64_t *tempty = tfull + 2;
    uint64_t *final_bar = tempty + 2;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(final_bar + 1);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = args.T, ng = args.n_groups;
    const int n_tiles = (T + BM - 1) / BM;
    const int k_blocks = args.D / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < n_stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], epi_warps<R>());
        }
        mbar_init(final_bar, 1);
        *s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW1);
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, C::TMEM_COLS);
        tmem_relinquish();
    }
    // W2 into shared memory (2 ng rows of R bf16), 16 bytes per thread and step
    {
        const int n16 = w2_bytes / 16;
        const uint4 *src = reinterpret_cast<const uint4 *>(args.W2);
        uint4 *dst = reinterpret_cast<uint4 *>(w2s);
        for (int i = threadIdx.x; i < n16; i += router_threads<R>()) dst[i] = src[i];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;

    if (warp == 0) {
        // ===================== TMA producer =====================
        int stage = 0;
        uint32_t phase = 0, used = 0, last_parity = 0;
        for (int tile = blockIdx.x; tile < n_tiles && !*s_abort; tile += gridDim.x) {
            for (int kb = 0; kb < k_blocks; ++kb) {
                int ok = 1;
                if (lane == 0) ok = mbar_wait(&empty[stage], phase ^ 1u, args.status);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) { *s_abort = 1; break; }
                if (lane == 0) {
                    uint8_t *sa = stages + stage * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                    tma_load_2d(sa, &tmX, &full[stage], kb * BK, tile * BM);
                    tma_load_2d(sa + C::A_BYTES, &tmW1, &full[stage], kb * BK, 0);
                }
                used |= 1u << stage;
                last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == n_stages) { stage = 0; phase ^= 1u; }
            }
        }
        if (lane == 0)
            for (int s = 0; s < n_stages; ++s)
                if (used & (1u << s)) mbar_wait(&full[s], (last_parity >> s) & 1u, args.status);
        __syncwarp();
    } else if (warp == 1) {
        // ===================== tcgen05 issuer =====================
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int tile = blockIdx.x; tile < n_tiles && !*s_abort; tile += gridDim.x) {
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, args.status)) { *s_abort = 1; break; }
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * R);
                bool ok = true;
                for (int kb = 0; kb < k_blocks; ++kb) {
                    if (!mbar_wait(&full[stage], phase, args.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(stages + stage * C::STAGE_BYTES);
                    const uint32_t b0 = a0 + C::A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_bf16(d, sw128_kmajor_desc(a0 + kk * 32), sw128_kmajor_desc(b0 + kk * 32),
                                 C::IDESC, (kb | kk) != 0);
                    mma_commit(&empty[stage]);
                    if (++stage == n_stages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) { *s_abort = 1; break; }
                mma_commit(&tfull[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            mma_commit(final_bar);
            mbar_wait(final_bar, 0, args.status);
        }
        __syncwarp();
    } else {
        // ===================== epilogue (warps 2..9) =====================
        const int quad = warp & 3;      // TMEM lanes 32*quad .. 32*quad+31
        constexpr int kParts = epi_warps<R>() / 4;
        const int part = (warp - 2) >> 2;  // which share of the groups
        const int row = quad * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        const bool words = (ng & 3) == 0;  // mask rows start on 4-byte boundaries
        // shares of a multiple of 4 groups: word stores never straddle two shares
        const int g_chunk = ((ng + 4 * kParts - 1) / (4 * kParts)) * 4;
        const int g_lo = min(ng, part * g_chunk);
        const int g_hi = part == kParts - 1 ? ng : min(ng, (part + 1) * g_chunk);
        for (int tile = blockIdx.x; tile < n_tiles && !*s_abort; tile += gridDim.x) {
            int ok = 1;
            if (lane == 0) ok = mbar_wait(&tfull[acc], acc_phase, args.status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) { *s_abort = 1; break; }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                   static_cast<uint32_t>(acc * R);
            float z[R];
#pragma unroll
            for (int c = 0; c < R; c += 16) {
                uint32_t v[16];
                tmem_ld16(taddr + c, v);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 16; ++q) z[c + q] = __uint_as_float(v[q]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);  // the next tile may reuse this accumulator
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }

            const int t = tile * BM + row;
            const bool valid = t < T;
            if (!REORDER && !valid) continue;
            // the tile's ballots, [tile][g][quad], for the fused reorder
            uint32_t *bal = REORDER ? partition_ws(args.ws, n_tiles, ng).bal + static_cast<size_t>(tile) * ng * 4
                                    : nullptr;
            uint8_t *mrow = args.mask + static_cast<size_t>(t) * ng;
            float *lrow = args.logits != nullptr ? args.logits + static_cast<size_t>(t) * 2 * ng : nullptr;
            for (int g0 = g_lo; g0 < g_hi; g0 += 4) {
                // logits of groups g0..g0+3 (8 FMA chains, each in ascending j)
                float acc8[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) acc8[q] = 0.f;
                const int nrow = min(8, 2 * (g_hi - g0));
#pragma unroll
                for (int c = 0; c < R / 8; ++c) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        if (q >= nrow) break;
                        const uint4 w = reinterpret_cast<const uint4 *>(w2s + (2 * g0 + q) * R)[c];
                        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            acc8[q] = fmaf(z[8 * c + 2 * e], __uint_as_float(ww[e] << 16), acc8[q]);
                            acc8[q] = fmaf(z[8 * c + 2 * e + 1], __uint_as_float(ww[e] & 0xFFFF0000u), acc8[q]);
                        }
                    }
                }
                uint32_t word = 0;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int g = g0 + u;
                    if (g >= g_hi) break;
                    const float r0 = acc8[2 * u], r1 = acc8[2 * u + 1];
                    const uint32_t m = r0 >= r1 ? 1u : 0u;  // argmax over (r0, r1): ties go to class 0
                    if (REORDER) {
                        const uint32_t b = __ballot_sync(0xffffffffu, valid && m != 0u);
                        if (lane == 0) bal[g * 4 + quad] = b;
                    }
                    if (!valid) continue;
                    if (lrow != nullptr) *reinterpret_cast<float2 *>(lrow + 2 * g) = make_float2(r0, r1);
                    if (words) word |= m << (8 * u);
                    else mrow[g] = static_cast<uint8_t>(m);
                }
                if (words && valid) *reinterpret_cast<uint32_t *>(mrow + g0) = word;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
    if constexpr (REORDER) {
        static_assert(BM == kPartTile, "one ballot tile per router tile");
        __shared__ int warp_sums[32];
        __shared__ int s_total;
        __shared__ int s_ok;
        const PartitionWs w = partition_ws(args.ws, n_tiles, ng);
        // every CTA takes part in both barriers, also after a failure of its own
        const bool ok1 = grid_barrier(w.ctr, gridDim.x, args.status, &s_ok) && !*s_abort;
        if (ok1) partition_scan(w, n_tiles, ng, args.counts, warp_sums, &s_total);
        const bool ok2 = grid_barrier(w.ctr, 2u * gridDim.x, args.status, &s_ok);
        if (!ok1 || !ok2) return;
        // the tile's ballots and offsets are staged in the (now idle) pipeline stages
        partition_place(w, n_tiles, ng, T, args.counts, args.perm, stages);
    }
}

template <int R, bool REORDER = false>
cudaError_t launch_t(const CUtensorMap &tmX, const CUtensorMap &tmW1, const RouterArgs &a, int num_sms,
                     cudaStream_t s) {
    using C = RouterCfg<R>;
    auto kern = router_kernel<R, REORDER>;
    const int w2_bytes = 2 * a.n_groups * R * 2;
    const int smem = C::smem_bytes(w2_bytes);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    RouterArgs args = a;
    args.stages = C::stages(w2_bytes);
    const int tiles = (a.T + BM - 1) / BM;
    const int grid = tiles < num_sms ? tiles : num_sms;  // one CTA per SM at most: all resident
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(router_threads<R>());
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = REORDER ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, tmX, tmW1, args);
}

// ---------------------------------------------------------------------------
// Decode router (T <= 16 tokens) on CUDA cores: a cluster of kDecSplit CTAs
// per token.  CTA k forms partial z[j] over its slice of d (warp w takes
// j = w, w + 8, ...; lanes split the slice, 16-byte loads, fixed-order warp
// reduction); after a cluster barrier CTA 0 adds the partials in rank order
// through distributed shared memory and forms the logits exactly as the
// tensor-core path's epilogue does (fp32 FMAs in ascending j, ties to class 0).
constexpr int kDecThreads = 256;
constexpr int kDecSplit = 8;

__global__ void __cluster_dims__(kDecSplit, 1, 1) __launch_bounds__(kDecThreads)
    router_decode_kernel(const uint16_t *__restrict__ X, const uint16_t *__restrict__ W1,
                         const RouterArgs a) {
    __shared__ float zs[64];  // r <= 64 partial sums of this CTA's slice
    // Every CTA reads its peers' shared memory: without the cluster this
    // kernel is compiled for (a launch that dropped the cluster shape) there
    // are no peers, so record the error, write nothing and touch no peer.
    if (cluster_nctarank() != kDecSplit) {
        if (threadIdx.x == 0 && a.status != nullptr) atomicCAS(a.status, 0, kStatusLaunch);
        return;
    }
    const int t = blockIdx.x / kDecSplit;
    const uint32_t rank = cluster_ctarank();
    const int D = a.D, r = a.r;
    const int slice = D / kDecSplit;  // D % 512 == 0, so slices are whole 16-byte chunks
    const int d0 = static_cast<int>(rank) * slice;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint4 *xrow = reinterpret_cast<const uint4 *>(X + static_cast<size_t>(t) * D + d0);
    for (int j = warp; j < r; j += kDecThreads / 32) {
        const uint4 *wrow = reinterpret_cast<const uint4 *>(W1 + static_cast<size_t>(j) * D + d0);
        float acc = 0.f;
        for (int c = lane; c < slice / 8; c += 32) {
            const uint4 wv = wrow[c], xv = xrow[c];
            const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w}, xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc = fmaf(__uint_as_float(xw[e] << 16), __uint_as_float(ww[e] << 16), acc);
                acc = fmaf(__uint_as_float(xw[e] & 0xFFFF0000u), __uint_as_float(ww[e] & 0xFFFF0000u), acc);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) zs[j] = acc;
    }
    cluster_sync();  // every CTA's partial z is in its shared memory
    if (rank == 0) {
        __shared__ float z[64];
        for (int j = threadIdx.x; j < r; j += kDecThreads) {
            float v = 0.f;
            for (uint32_t k = 0; k < kDecSplit; ++k) v += ld_shared_cluster_f32(&zs[j], k);
            z[j] = v;
        }
        __syncthreads();
        const int ng = a.n_groups;
        for (int g = threadIdx.x; g < ng; g += kDecThreads) {
            const uint16_t *w0 = a.W2 + static_cast<size_t>(2 * g) * r;
            const uint16_t *w1 = w0 + r;
            float r0 = 0.f, r1 = 0.f;
            for (int j = 0; j < r; ++j) {
                r0 = fmaf(z[j], __uint_as_float(static_cast<uint32_t>(w0[j]) << 16), r0);
                r1 = fmaf(z[j], __uint_as_float(static_cast<uint32_t>(w1[j]) << 16), r1);
            }
            a.mask[static_cast<size_t>(t) * ng + g] = r0 >= r1 ? 1 : 0;  // ties go to class 0
            if (a.logits != nullptr)
                *reinterpret_cast<float2 *>(a.logits + static_cast<size_t>(t) * 2 * ng + 2 * g) = make_float2(r0, r1);
        }
    }
    cluster_sync();  // the other CTAs' shared memory is read until here
}

}  // namespace

cudaError_t launch_router_decode(const uint16_t *X, const uint16_t *W1, const RouterArgs &a,
                                 cudaStream_t s) {
    router_decode_kernel<<<a.T * kDecSplit, kDecThreads, 0, s>>>(X, W1, a);
    return cudaGetLastError();
}

bool router_supported(int r, int n_groups) {
    if (r != 16 && r != 32 && r != 64) return false;
    return n_groups >= 1 && 2 * n_groups * r * 2 <= kW2MaxBytes;
}

size_t route_reorder_workspace_bytes(int T, int n_groups) { return partition_workspace_bytes(T, n_groups); }

cudaError_t launch_route_reorder(const CUtensorMap &tmX, const CUtensorMap &tmW1, const RouterArgs &a,
                                 int num_sms, cudaStream_t s) {
    if (a.r == 16) return launch_t<16, true>(tmX, tmW1, a, num_sms, s);
    if (a.r == 32) return launch_t<32, true>(tmX, tmW1, a, num_sms, s);
    if (a.r == 64) return launch_t<64, true>(tmX, tmW1, a, num_sms, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_router(const CUtensorMap &tmX, const CUtensorMap &tmW1, const RouterArgs &a,
                          int num_sms, cudaStream_t s) {
    if (a.r == 16) return launch_t<16>(tmX, tmW1, a, num_sms, s);
    if (a.r == 32) return launch_t<32>(tmX, tmW1, a, num_sms, s);
    if (a.r == 64) return launch_t<64>(tmX, tmW1, a, num_sms, s);
    return cudaErrorInvalidValue;
}

}  // namespace wide
