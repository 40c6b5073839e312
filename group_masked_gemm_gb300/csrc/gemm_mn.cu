// gemm_mn.cu -- GEMM-MN on tcgen05 (WIDE, App. B "Implementation of
// GEMM-MN", Algorithm 2; Sec. 3.1 Eq. 2 and Eq. 3).
//
//   out[t, n] = M[t, n/G] * f( sum_k A[t,k] B[n,k] )
//
// with f = identity (q_proj) or the fused silu(gate) * up (FFN gate/up, where
// B stacks the matching rows of W_gate and W_up).  Rows are consumed in the
// reordered order of each routing column: the active tokens of group g are
// perm[g][0 .. counts[g]).
//
// GB300 design (one persistent CTA per SM, 10 warps):
//   warp 0      TMA producer of the weight tile of the group (dense, tiled
//               TMA, 128-byte swizzle).
//   warps 6..9  gather the A rows (token rows picked through perm) with
//               16-byte cp.async copies written straight into the
//               128-byte-swizzled layout the UMMA descriptor expects, one
//               128-byte row segment per 8 lanes; only the rows that hold
//               active tokens are copied (the l=1 predicate of Eq. 20).
//               Measured on GB300, the TMA row gather (tile::gather4) issues
//               at ~80 clocks per 4-row instruction whichever lanes issue it,
//               ~6 B/clk per SM against the ~58 B/clk the MMA consumes, so the
//               gather goes through the load/store path instead.
//   warp 1      TMEM owner and single-thread tcgen05.mma issuer
//               (M = 128 gathered rows, N = 2 x 128 for gate/up, K = 16 per
//               instruction, fp32 accumulators in TMEM, double buffered).
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, activation, bf16
//               conversion, scatter of each row to its token (perm), zeros for
//               the inactive rows of the boundary tile.
// The work list is built in shared memory from counts[]: a tile of group g
// exists only for row offsets below counts[g] (the l=0 CTA-level predicate
// becomes "never scheduled"), followed by "zero tiles" that write the exact
// zeros of the inactive (token, group) blocks.  Compute tiles are ordered by
// (token band, group, tile): each group's tiles are split into `bands`
// consecutive ranges, and since a group's active tokens are sorted, range b
// of every group covers about the same band of token rows.  CTAs running at
// the same time then share one band of X (sized to stay resident in L2) and
// the weights of a few groups, instead of sweeping all of X for each group.
#include "common.cuh"
#include "internal.h"

namespace wide {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // one 128-byte swizzle row of bf16
constexpr int kGatherWarps = 4;                    // A-row gather warps 6..9
constexpr int kThreads = 32 * (6 + kGatherWarps);  // producer, MMA, 4 epilogue, 4 gather
constexpr int kSmemBudget = 225 * 1024;

template <MNMode MODE, int BN_OP>
struct Cfg {
    static constexpr int N_MMA = (MODE == MNMode::kGateUp) ? 2 * BN_OP : BN_OP;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = N_MMA * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SCHED_BYTES = (3 * kMaxGroups + 2) * 4;
    static constexpr int BAR_BYTES = 256;
    static constexpr int STAGES_FIT = (kSmemBudget - 1024 - SCHED_BYTES - BAR_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr int TMEM_COLS = (2 * N_MMA <= 64) ? 64
                                    : (2 * N_MMA <= 128) ? 128
                                    : (2 * N_MMA <= 256) ? 256 : 512;
    static constexpr uint32_t IDESC = idesc_bf16_f32(BM, N_MMA);
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + SCHED_BYTES + BAR_BYTES;
    static_assert(STAGES >= 2, "pipeline needs two stages");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

struct Sched {
    int *cpre;    // [bands*ng+1] prefix of compute items per (band, group)
    int *zpre;    // [ng+1] prefix of zero items per group
    int *counts;  // [ng]
    int ng, nsub, bands, n_compute, n_total;
};

// First tile of band b for a group with mt tiles: ceil(b * mt / bands).
__device__ __forceinline__ int band_lo(int b, int mt, int bands) {
    return (b * mt + bands - 1) / bands;
}

struct Item {
    int g, m, ns;  // group, 128-row tile of the reordered column, N sub-tile
    bool zero;     // a zero-fill tile (rows m*128.. of the inactive part)
};

__device__ __forceinline__ int upper_group(const int *pre, int ng, int i) {
    int lo = 0, hi = ng;  // largest g with pre[g] <= i
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= i) lo = mid;
        else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ Item decode_item(const Sched &s, int i) {
    Item it;
    if (i < s.n_compute) {
        const int e = upper_group(s.cpre, s.bands * s.ng, i);  // entry (band, group)
        const int b = e / s.ng;
        it.g = e - b * s.ng;
        const int local = i - s.cpre[e];
        const int mt = (s.counts[it.g] + BM - 1) / BM;
        const int q = local / s.nsub;
        it.m = band_lo(b, mt, s.bands) + q;
        it.ns = local - q * s.nsub;
        it.zero = false;
    } else {
        const int zi = i - s.n_compute;
        it.g = upper_group(s.zpre, s.ng, zi);
        const int first_zero_tile = (s.counts[it.g] + BM - 1) / BM;
        it.m = first_zero_tile + (zi - s.zpre[it.g]);
        it.ns = 0;
        it.zero = true;
    }
    return it;
}

// Warp 0 scans the per-group item counts held in pre[1..ng] into prefixes.
__device__ __forceinline__ void warp_prefix(int *pre, int ng) {
    const int lane = threadIdx.x & 31;
    const int per = (ng + 31) / 32;
    const int lo = min(ng, lane * per), hi = min(ng, lo + per);
    int sum = 0;
    for (int g = lo; g < hi; ++g) sum += pre[g + 1];
    int inc = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += y;
    }
    int run = inc - sum;
    for (int g = lo; g < hi; ++g) {
        run += pre[g + 1];
        pre[g + 1] = run;
    }
    if (lane == 0) pre[0] = 0;
}

__device__ __forceinline__ float silu_mul(float gate, float up) {
    return __fdividef(gate, 1.0f + __expf(-gate)) * up;
}

template <MNMode MODE, int BN_OP>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_mn_kernel(const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                   const MNArgs args) {
    using C = Cfg<MODE, BN_OP>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *stages = smem;
    int *s_cpre = reinterpret_cast<int *>(smem + C::STAGES * C::STAGE_BYTES);
    int *s_zpre = s_cpre + (kMaxGroups + 1);
    int *s_counts = s_zpre + (kMaxGroups + 1);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::STAGES * C::STAGE_BYTES + C::SCHED_BYTES);
    uint64_t *full = bars;                    // [STAGES] TMA -> MMA
    uint64_t *empty = bars + C::STAGES;       // [STAGES] MMA -> TMA
    uint64_t *tfull = bars + 2 * C::STAGES;   // [2] MMA -> epilogue
    uint64_t *tempty = tfull + 2;             // [2] epilogue -> MMA
    uint64_t *final_bar = tempty + 2;         // MMA drain
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(final_bar + 1);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = args.T;
    const int ng = args.n_out / args.G;

    // ---- schedule: tiles of each group exist only below counts[g] ---------
    const int bands = args.bands;
    const int nsub = args.G / BN_OP;
    for (int g = threadIdx.x; g < ng; g += kThreads) {
        const int c = ld_nc_s32(args.counts + g);
        s_counts[g] = c;
        const int mt = (c + BM - 1) / BM;
        const int covered = mt * BM;
        s_zpre[g + 1] = covered < T ? (T - covered + BM - 1) / BM : 0;
        for (int b = 0; b < bands; ++b)
            s_cpre[b * ng + g + 1] = (band_lo(b + 1, mt, bands) - band_lo(b, mt, bands)) * nsub;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            // producer's expect_tx arrival + one per gather thread once its copies landed
            mbar_init(&full[s], 1 + 32 * kGatherWarps);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);
        }
        mbar_init(final_bar, 1);
        *s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmB0);
        if (MODE == MNMode::kGateUp) prefetch_tmap(&tmB1);
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, C::TMEM_COLS);
        tmem_relinquish();
    }
    __syncthreads();
    if (warp == 0) warp_prefix(s_cpre, bands * ng);
    if (warp == 1) warp_prefix(s_zpre, ng);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    Sched sch;
    sch.cpre = s_cpre;
    sch.zpre = s_zpre;
    sch.counts = s_counts;
    sch.ng = ng;
    sch.nsub = nsub;
    sch.bands = bands;
    sch.n_compute = s_cpre[bands * ng];
    sch.n_total = sch.n_compute + s_zpre[ng];
    const uint32_t tmem_base = *s_tmem;
    const int k_blocks = args.K / BK;

    if (warp == 0) {
        // ===================== TMA producer =====================
        int stage = 0;
        uint32_t phase = 0;
        uint32_t used = 0, last_parity = 0;  // per-stage bookkeeping for the drain
        for (int i = blockIdx.x; i < sch.n_total && !*s_abort; i += gridDim.x) {
            const Item it = decode_item(sch, i);
            if (it.zero) continue;
            const uint32_t bytes = static_cast<uint32_t>(C::B_BYTES);
            const int nrow = it.g * args.G + it.ns * BN_OP;
            for (int kb = 0; kb < k_blocks; ++kb) {
                int ok = 1;
                if (lane == 0) ok = mbar_wait(&empty[stage], phase ^ 1u, args.status);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) { *s_abort = 1; break; }
                uint8_t *sb = stages + stage * C::STAGE_BYTES + C::A_BYTES;
                if (lane == 0) mbar_arrive_expect_tx(&full[stage], bytes);
                if (lane == 0) {
                    tma_load_2d(sb, &tmB0, &full[stage], kb * BK, nrow);
                    if (MODE == MNMode::kGateUp)
                        tma_load_2d(sb + BN_OP * BK * 2, &tmB1, &full[stage], kb * BK, nrow);
                }
                used |= 1u << stage;
                last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        // never leave the CTA with bulk copies still landing in its shared memory
        if (lane == 0)
            for (int s = 0; s < C::STAGES; ++s)
                if (used & (1u << s)) mbar_wait(&full[s], (last_parity >> s) & 1u, args.status);
        __syncwarp();
    } else if (warp == 1) {
        // ===================== tcgen05 issuer =====================
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int i = blockIdx.x; i < sch.n_total && !*s_abort; i += gridDim.x) {
                const Item it = decode_item(sch, i);
                if (it.zero) continue;
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, args.status)) { *s_abort = 1; break; }
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * C::N_MMA);
                bool ok = true;
                for (int kb = 0; kb < k_blocks; ++kb) {
                    if (!mbar_wait(&full[stage], phase, args.status)) { ok = false; break; }
                    fence_proxy_async_smem();  // A rows were written by cp.async (generic proxy)
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(stages + stage * C::STAGE_BYTES);
                    const uint32_t b0 = a0 + C::A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_bf16(d, sw128_kmajor_desc(a0 + kk * 32), sw128_kmajor_desc(b0 + kk * 32),
                                 C::IDESC, (kb | kk) != 0);
                    mma_commit(&empty[stage]);
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) { *s_abort = 1; break; }
                mma_commit(&tfull[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            mma_commit(final_bar);
            mbar_wait(final_bar, 0, args.status);
        }
        __syncwarp();
    } else if (warp >= 6) {
        // ===================== cp.async row gather (warps 6..9) =====================
        // Warp gw owns rows 32*gw .. 32*gw+31 of the A tile; one instruction
        // copies 4 rows x 128 bytes (8 lanes per row, 16 bytes per lane) into
        // the 128-byte-swizzled layout the UMMA descriptor expects.  Each
        // thread announces a stage on full[stage] with a non-incrementing
        // cp.async arrive, so no thread waits for its own copies; the MMA
        // thread makes them visible to the tensor core (proxy fence) after
        // acquiring the barrier.
        // The token indices of the next tile are loaded while the current
        // tile streams, so no tile starts with a dependent global load.
        const int gw = warp - 6;
        const int sub = lane >> 3, chunk = lane & 7;
        auto row_token = [&](int i) -> int {  // this lane's row of compute item i, or -1
            const Item it = decode_item(sch, i);
            const int rows_valid = min(BM, sch.counts[it.g] - it.m * BM);
            const int my_row = 32 * gw + lane;
            return my_row < rows_valid
                       ? ld_nc_s32(args.perm + static_cast<size_t>(it.g) * T + it.m * BM + my_row)
                       : -1;
        };
        int stage = 0;
        uint32_t phase = 0;
        // compute items are exactly i < n_compute (the zero-fill items follow them)
        int next_tok = blockIdx.x < sch.n_compute ? row_token(blockIdx.x) : -1;
        for (int i = blockIdx.x; i < sch.n_compute && !*s_abort; i += gridDim.x) {
            const int my_tok = next_tok;
            int toks[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) toks[q] = __shfl_sync(0xffffffffu, my_tok, 4 * q + sub);
            if (i + static_cast<int>(gridDim.x) < sch.n_compute) next_tok = row_token(i + gridDim.x);
            for (int kb = 0; kb < k_blocks; ++kb) {
                int ok = 1;
                if (lane == 0) ok = mbar_wait(&empty[stage], phase ^ 1u, args.status);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) { *s_abort = 1; break; }
                const uint32_t sa = smem_u32(stages + stage * C::STAGE_BYTES);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int row = 32 * gw + 4 * q + sub;
                    if (toks[q] >= 0) {
                        const uint16_t *src = args.a_rows + static_cast<size_t>(toks[q]) * args.K + kb * BK + chunk * 8;
                        cp_async16(sa + row * 128 + ((chunk ^ (row & 7)) << 4), src);
                    }
                }
                cp_async_mbar_arrive_noinc(&full[stage]);
                if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        cp_async_wait_all();
    } else {
        // ===================== epilogue (warps 2..5) =====================
        const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
        const int row = quad * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        // This CTA's items are i = blockIdx.x + k * gridDim.x: compute items
        // first (i < n_compute), then zero-fill items.  Zero-fill items need
        // only stores, so they are spread between the compute tiles'
        // epilogues, while the tensor core works on the next tile, instead of
        // being written after the last MMA.
        const int bx = static_cast<int>(blockIdx.x), grid = static_cast<int>(gridDim.x);
        const int n_comp_mine = sch.n_compute > bx ? (sch.n_compute - bx + grid - 1) / grid : 0;
        const int n_all_mine = sch.n_total > bx ? (sch.n_total - bx + grid - 1) / grid : 0;
        const int n_zero_mine = n_all_mine - n_comp_mine;
        const int zero_per_tile = n_comp_mine > 0 ? (n_zero_mine + n_comp_mine - 1) / n_comp_mine : n_zero_mine;
        int zk = 0;  // zero-fill items written so far
        auto write_zero_items = [&](int count) {
            for (int c = 0; c < count && zk < n_zero_mine; ++c, ++zk) {
                const Item it = decode_item(sch, bx + (n_comp_mine + zk) * grid);
                const int j = it.m * BM + row;
                if (j < T) {
                    const int token = ld_nc_s32(args.perm + static_cast<size_t>(it.g) * T + j);
                    uint16_t *orow = args.out + static_cast<size_t>(token) * args.n_out + it.g * args.G;
                    for (int cidx = 0; cidx < args.G; cidx += 8) st_global_cs_v4(orow + cidx, 0, 0, 0, 0);
                }
            }
        };
        for (int k = 0; k < n_comp_mine && !*s_abort; ++k) {
            write_zero_items(zero_per_tile);
            const Item it = decode_item(sch, bx + k * grid);
            const int32_t *pg = args.perm + static_cast<size_t>(it.g) * T;
            const int j = it.m * BM + row;
            const bool valid = j < T;
            const int token = valid ? ld_nc_s32(pg + j) : 0;
            uint16_t *orow = args.out + static_cast<size_t>(token) * args.n_out + it.g * args.G;
            const bool active = j < sch.counts[it.g];
            int ok = 1;
            if (lane == 0) ok = mbar_wait(&tfull[acc], acc_phase, args.status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) { *s_abort = 1; break; }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                   static_cast<uint32_t>(acc * C::N_MMA);
            uint16_t *dst = orow + it.ns * BN_OP;
#pragma unroll 1
            for (int cb = 0; cb < BN_OP; cb += 32) {
                uint32_t v[16];
                if (MODE == MNMode::kGateUp) {
                    uint32_t gr[32], ur[32];
                    tmem_ld32(taddr + cb, gr);
                    tmem_ld32(taddr + BN_OP + cb, ur);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const float h0 = silu_mul(__uint_as_float(gr[2 * q]), __uint_as_float(ur[2 * q]));
                        const float h1 = silu_mul(__uint_as_float(gr[2 * q + 1]), __uint_as_float(ur[2 * q + 1]));
                        v[q] = active ? pack_bf16x2(h0, h1) : 0u;
                    }
                } else {
                    uint32_t yr[32];
                    tmem_ld32(taddr + cb, yr);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        v[q] = active ? pack_bf16x2(__uint_as_float(yr[2 * q]), __uint_as_float(yr[2 * q + 1])) : 0u;
                }
                if (valid) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        st_global_cs_v4(dst + cb + 8 * q, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        if (!*s_abort) write_zero_items(n_zero_mine);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <MNMode MODE, int BN_OP>
cudaError_t launch_t(const CUtensorMap &tmB0, const CUtensorMap &tmB1, const MNArgs &a,
                     int num_sms, cudaStream_t s) {
    using C = Cfg<MODE, BN_OP>;
    auto kern = gemm_mn_kernel<MODE, BN_OP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<num_sms, kThreads, C::SMEM_BYTES, s>>>(tmB0, tmB1, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_mn(MNMode mode, int bn, const CUtensorMap &tmB0, const CUtensorMap &tmB1,
                           const MNArgs &a, int num_sms, cudaStream_t s) {
    if (mode == MNMode::kGateUp) {
        if (bn == 128) return launch_t<MNMode::kGateUp, 128>(tmB0, tmB1, a, num_sms, s);
        if (bn == 64) return launch_t<MNMode::kGateUp, 64>(tmB0, tmB1, a, num_sms, s);
    } else {
        if (bn == 256) return launch_t<MNMode::kPlain, 256>(tmB0, tmB1, a, num_sms, s);
        if (bn == 128) return launch_t<MNMode::kPlain, 128>(tmB0, tmB1, a, num_sms, s);
        if (bn == 64) return launch_t<MNMode::kPlain, 64>(tmB0, tmB1, a, num_sms, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace wide
