// gemm_k.cu -- GEMM-K on tcgen05 (WIDE, App. B "Implementation of GEMM-K",
// Eq. 21; Sec. 3.1 Eq. 2-3 for o_proj / down_proj).
//
//   Y[t, n] = sum_g M[t,g] sum_{k in [gG,(g+1)G)} A[t,k] W[n,k]
//
// GB300 design: a persistent CTA owns an output tile of 128 tokens (natural
// order) x BN columns and keeps its fp32 accumulator in TMEM for the whole
// reduction, adding the groups in ascending order -- a per-token ordered
// reduction with no atomics and a deterministic result (a workspace only for
// the split cases below).  The
// routing mask is applied inside the tensor core: every tcgen05.mma of group
// g carries a disable-output-lane mask whose bit is set for the tokens of the
// tile with M[t,g] = 0, so their accumulator rows are left untouched (the
// l=2 predicate of Eq. 20, per TMEM lane).  A group with no active token in
// the tile is skipped entirely (copies, MMAs and barriers; the l=0
// predicate), and values of A inside inactive groups never reach Y.
//
// Warps: 0 TMA producer, 1 TMEM owner + MMA issuer, 2 mask builder (turns the
// tile's mask block into lane masks and a list of live groups, double
// buffered), 3..6 epilogue (TMEM -> bf16 rows of Y, then re-zeroes the
// accumulator for its next tile).
//
// Decode (T <= 16) runs the same kernel with a 16-row token stage (AR = 16):
// a stage holds 2 KB of tokens and 16 KB of weights, so 11 stages of weights
// are in flight per SM.  The M = 128 MMA still reads 128 A rows; rows 16..127
// fall inside the same stage's weight tile and land in TMEM lanes that the
// lane mask disables (tokens >= T are inactive in every group).  The groups
// live for some token are dealt in equal contiguous shares to `splits` work
// items per output tile (so a sparse mask does not leave a few CTAs with most
// of the live weights); each item writes fp32 partial sums, added in split
// order by a finalize kernel.
//
// Prefill takes tiles round-robin, so its last wave holds items mod
// num_SMs tiles.  When that wave would leave at least half of the SMs idle
// and the caller passed the optional workspace, each of its tiles is cut
// into equal shares of its live groups (the tail split): the shares write
// fp32 partials to a compact array, and gemm_k_tail_finalize_kernel adds
// them in share order.
#include "common.cuh"
#include "internal.h"

namespace wide {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kThreads = 224;
constexpr int kMaxKGroups = 512;
constexpr int kSmemBudget = 225 * 1024;

template <int BN, int AR>
struct KCfg {
    static_assert(AR == BM || AR == 16, "token stage rows");
    static constexpr int A_BYTES = AR * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    // per mask buffer: lane masks [ng][4] + live-group list [ng] + count
    static constexpr int MASK_BUF_BYTES = kMaxKGroups * 16 + kMaxKGroups * 4 + 16;
    static constexpr int BAR_BYTES = 512;
    static constexpr int STAGES_FIT =
        (kSmemBudget - 1024 - 2 * MASK_BUF_BYTES - BAR_BYTES) / STAGE_BYTES;
    static constexpr int MAX_STAGES = AR == BM ? 8 : 12;
    static constexpr int STAGES = STAGES_FIT > MAX_STAGES ? MAX_STAGES : STAGES_FIT;
    static constexpr int TMEM_COLS = (2 * BN <= 256) ? 256 : 512;
    static constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 2 * MASK_BUF_BYTES + BAR_BYTES;
    static_assert(STAGES >= 2, "pipeline needs two stages");
    static_assert((2 * STAGES + 9) * 8 + 8 <= BAR_BYTES, "barrier area");
    static_assert(STAGE_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "SW128 operand alignment");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// Mask buffer b (of 2) inside the mask area: lane masks [ng][4], the live
// group list [ng], and the slice live[first, first + n_live) of this item.
struct MaskBuf {
    uint32_t *lanes;  // [ng][4] disable-output-lane words
    int *live;        // [ng] live groups, ascending
    int *n_live;
    int *first;
};

template <int BUF_BYTES>
__device__ __forceinline__ MaskBuf mask_buf(uint8_t *area, int b) {
    uint8_t *base = area + b * BUF_BYTES;
    return MaskBuf{reinterpret_cast<uint32_t *>(base), reinterpret_cast<int *>(base + kMaxKGroups * 16),
                   reinterpret_cast<int *>(base + kMaxKGroups * 20),
                   reinterpret_cast<int *>(base + kMaxKGroups * 20 + 4)};
}

// Decode lane masks (T <= 16 tokens in lanes 0..15 of the tile): lane i of the
// warp takes group g0 + i, reads its mask byte for every token (one coalesced
// 32-byte row segment per token) and forms the word of active tokens; lanes
// 32..127 of the tile are always disabled.  Returns the number of live groups.
__device__ __forceinline__ int build_decode_masks(const uint8_t *__restrict__ mask, int T, int ng,
                                                  uint32_t *lanes, int *live) {
    const int lane = threadIdx.x & 31;
    int n_live = 0;
    for (int g0 = 0; g0 < ng; g0 += 32) {
        const int g = g0 + lane;
        uint32_t word = 0;
        if (g < ng) {
            uint8_t v[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) v[t] = t < T ? mask[static_cast<size_t>(t) * ng + g] : 0;
#pragma unroll
            for (int t = 0; t < 16; ++t) word |= (v[t] != 0 ? 1u : 0u) << t;
            *reinterpret_cast<uint4 *>(lanes + g * 4) = make_uint4(~word, ~0u, ~0u, ~0u);
        }
        const uint32_t b = __ballot_sync(0xffffffffu, word != 0u);
        if (word != 0u) live[n_live + __popc(b & ((1u << lane) - 1u))] = g;
        n_live += __popc(b);
    }
    return n_live;
}


// Lane masks and live-group list of one tile of Q*32 tokens starting at m0:
// for every group g, word q (q < Q) has bit i set when token m0+32q+i is
// INACTIVE (or beyond T); the group is live when any token is active.  Runs
// on one warp.  When n_groups is a multiple of 16 each lane reads 16 groups
// of a token row with one 16-byte load.
template <int Q>
__device__ __forceinline__ int build_tile_masks(const uint8_t *__restrict__ mask, int T, int ng,
                                                int m0, uint32_t *lanes, int *live) {
    const int lane = threadIdx.x & 31;
    int n_live = 0;
    auto emit = [&](int g, const uint32_t (&w)[Q]) {
        uint32_t mine = 0, any = 0;
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            any |= w[q];
            if (lane == q) mine = w[q];
        }
        if (lane < Q) lanes[g * Q + lane] = ~mine;
        if (any != 0u) {
            if (lane == 0) live[n_live] = g;
            ++n_live;
        }
    };
    if ((ng & 15) == 0) {
        // 16-byte loads of 16 groups; the loads of the next 16 groups are
        // issued before the current ones are used.
        auto load16 = [&](int g0, uint4 (&v)[Q]) {
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                const int t = m0 + 32 * q + lane;
                v[q] = t < T ? *reinterpret_cast<const uint4 *>(mask + static_cast<size_t>(t) * ng + g0)
                             : make_uint4(0, 0, 0, 0);
            }
        };
        uint4 v[Q];
        load16(0, v);
        for (int g0 = 0; g0 < ng; g0 += 16) {
            uint4 nv[Q];
            const bool more = g0 + 16 < ng;
            if (more) load16(g0 + 16, nv);
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                uint32_t w[Q];
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    const uint32_t word = u < 4 ? v[q].x : u < 8 ? v[q].y : u < 12 ? v[q].z : v[q].w;
                    w[q] = __ballot_sync(0xffffffffu, ((word >> ((u & 3) * 8)) & 0xFFu) != 0u);
                }
                emit(g0 + u, w);
            }
            if (more) {
#pragma unroll
                for (int q = 0; q < Q; ++q) v[q] = nv[q];
            }
        }
    } else {
        constexpr int kU = 4;
        for (int g0 = 0; g0 < ng; g0 += kU) {
            uint8_t v[kU][Q];
#pragma unroll
            for (int u = 0; u < kU; ++u)
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    const int t = m0 + 32 * q + lane;
                    const int g = g0 + u;
                    v[u][q] = (t < T && g < ng) ? mask[static_cast<size_t>(t) * ng + g] : 0;
                }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                if (g0 + u >= ng) break;
                uint32_t w[Q];
#pragma unroll
                for (int q = 0; q < Q; ++q) w[q] = __ballot_sync(0xffffffffu, v[u][q] != 0);
                emit(g0 + u, w);
            }
        }
    }
    return n_live;
}

// Work unit i of the persistent grid: output tile (mt, nt), share sp of nsp
// equal shares of the tile's live groups, and its tail-partial slot (-1: the
// unit writes Y, or the [splits][T][N] partial planes of a split launch).
struct KUnit {
    int mt, nt, sp, nsp, slot;
};

__device__ __forceinline__ KUnit k_unit(int i, int n_tiles, const KArgs &a) {
    KUnit u;
    if (a.n_direct < 0) {
        u.mt = i / (n_tiles * a.splits);
        const int rem = i - u.mt * n_tiles * a.splits;
        u.sp = rem / n_tiles;
        u.nt = rem - u.sp * n_tiles;
        u.nsp = a.splits;
        u.slot = -1;
    } else if (i < a.n_direct) {
        u.mt = i / n_tiles;
        u.nt = i - u.mt * n_tiles;
        u.sp = 0;
        u.nsp = 1;
        u.slot = -1;
    } else {
        const int j = i - a.n_direct;
        const int item = a.n_direct + j / a.tail_splits;
        u.mt = item / n_tiles;
        u.nt = item - u.mt * n_tiles;
        u.sp = j - (j / a.tail_splits) * a.tail_splits;
        u.nsp = a.tail_splits;
        u.slot = j;
    }
    return u;
}

__host__ __device__ __forceinline__ int k_units(int m_tiles, int n_tiles, const KArgs &a) {
    return a.n_direct < 0 ? m_tiles * n_tiles * a.splits
                          : a.n_direct + (m_tiles * n_tiles - a.n_direct) * a.tail_splits;
}

template <int BN, int AR>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_k_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const KArgs args) {
    using C = KCfg<BN, AR>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *stages = smem;
    uint8_t *mask_area = smem + C::STAGES * C::STAGE_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(mask_area + 2 * C::MASK_BUF_BYTES);
    uint64_t *full = bars;
    uint64_t *empty = bars + C::STAGES;
    uint64_t *tfull = bars + 2 * C::STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *mfull = tempty + 2;   // mask builder -> producer + MMA
    uint64_t *mempty = mfull + 2;   // producer + MMA -> mask builder
    uint64_t *final_bar = mempty + 2;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(final_bar + 1);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = args.T;
    const int ng = args.K / args.G;
    const int m_tiles = (T + BM - 1) / BM;
    const int n_tiles = args.N / BN;
    const int n_items = k_units(m_tiles, n_tiles, args);
    const int kb_per_group = args.G / BK;
    const bool partial_out = args.partial != nullptr;
    const uint32_t stage_bytes = static_cast<uint32_t>(args.a_rows * BK * 2 + C::B_BYTES);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);
            mbar_init(&mfull[b], 1);
            mbar_init(&mempty[b], 2);
        }
        mbar_init(final_bar, 1);
        *s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, C::TMEM_COLS);
        tmem_relinquish();
    }
    // the split-partial finalize (launched as a programmatic dependent) may
    // be scheduled now; it waits for this grid before reading the partials
    griddep_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    // Everything above touches no input or output.  The decode variant is
    // launched as a programmatic dependent of the kernel before it, so its
    // launch and set-up overlap that kernel's tail; every read of an input
    // and every write of an output comes after this wait.
    griddep_wait();
    // Accumulators start at zero: every MMA accumulates (lanes it skips must
    // keep the value of the groups already added).  Only the MMA issuer waits
    // for the zeroing (named barrier 1: warps 1, 3..6); the producer and the
    // mask builder start on the first tile at once.
    if (warp >= 3) {
        const int quad = warp & 3;
        uint32_t z[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) z[q] = 0u;
        for (int col = 0; col < 2 * BN; col += 32)
            tmem_st32(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + col, z);
        tmem_st_wait();
    }
    if (warp == 1 || warp >= 3) {
        tc_fence_before();
        named_barrier_sync(1, 5 * 32);
        tc_fence_after();
    }

    if (warp == 2) {
        // ===================== mask builder =====================
        int b = 0;
        uint32_t bphase = 0;
        for (int i = blockIdx.x; i < n_items && !*s_abort; i += gridDim.x) {
            const KUnit u = k_unit(i, n_tiles, args);
            const int m0 = u.mt * BM;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(&mempty[b], bphase ^ 1u, args.status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) { *s_abort = 1; break; }
            const MaskBuf mbuf = mask_buf<C::MASK_BUF_BYTES>(mask_area, b);
            int n_all;
            if constexpr (AR == BM) {
                n_all = build_tile_masks<4>(args.mask, T, ng, m0, mbuf.lanes, mbuf.live);
            } else {
                n_all = build_decode_masks(args.mask, T, ng, mbuf.lanes, mbuf.live);
            }
            // equal contiguous shares of the tile's live groups, one per split
            const int per = (n_all + u.nsp - 1) / u.nsp;
            const int first = min(n_all, u.sp * per);
            const int n_live = min(n_all, first + per) - first;
            if (lane == 0) {
                *mbuf.n_live = n_live;
                *mbuf.first = first;
            }
            __threadfence_block();
            __syncwarp();
            if (lane == 0) mbar_arrive(&mfull[b]);  // release semantics publish the buffer
            if (++b == 2) { b = 0; bphase ^= 1u; }
        }
    } else if (warp == 0) {
        // ===================== TMA producer =====================
        int stage = 0;
        uint32_t phase = 0;
        uint32_t used = 0, last_parity = 0;
        int b = 0;
        uint32_t bphase = 0;
        for (int i = blockIdx.x; i < n_items && !*s_abort; i += gridDim.x) {
            const KUnit u = k_unit(i, n_tiles, args);
            const int mt = u.mt, nt = u.nt;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(&mfull[b], bphase, args.status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) { *s_abort = 1; break; }
            const MaskBuf mbuf = mask_buf<C::MASK_BUF_BYTES>(mask_area, b);
            const int n_live = *mbuf.n_live;
            const int *live = mbuf.live + *mbuf.first;
            for (int li = 0; li < n_live && ok; ++li) {
                const int g = live[li];
                for (int kb = 0; kb < kb_per_group; ++kb) {
                    if (lane == 0) ok = mbar_wait(&empty[stage], phase ^ 1u, args.status);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    if (lane == 0) {
                        uint8_t *sa = stages + stage * C::STAGE_BYTES;
                        mbar_arrive_expect_tx(&full[stage], stage_bytes);
                        const int kx = g * args.G + kb * BK;
                        tma_load_2d(sa, &tmA, &full[stage], kx, mt * BM);
                        tma_load_2d(sa + C::A_BYTES, &tmB, &full[stage], kx, nt * BN);
                    }
                    used |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) { *s_abort = 1; break; }
            __syncwarp();
            if (lane == 0) mbar_arrive(&mempty[b]);
            if (++b == 2) { b = 0; bphase ^= 1u; }
        }
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
            int b = 0;
            uint32_t bphase = 0;
            for (int i = blockIdx.x; i < n_items && !*s_abort; i += gridDim.x) {
                if (!mbar_wait(&mfull[b], bphase, args.status)) { *s_abort = 1; break; }
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, args.status)) { *s_abort = 1; break; }
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
                const MaskBuf mbuf = mask_buf<C::MASK_BUF_BYTES>(mask_area, b);
                const int n_live = *mbuf.n_live;
                const int *live = mbuf.live + *mbuf.first;
                bool ok = true;
                for (int li = 0; li < n_live && ok; ++li) {
                    const int g = live[li];
                    const uint32_t l0 = mbuf.lanes[g * 4 + 0], l1 = mbuf.lanes[g * 4 + 1];
                    const uint32_t l2 = mbuf.lanes[g * 4 + 2], l3 = mbuf.lanes[g * 4 + 3];
                    for (int kb = 0; kb < kb_per_group; ++kb) {
                        if (!mbar_wait(&full[stage], phase, args.status)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t a0 = smem_u32(stages + stage * C::STAGE_BYTES);
                        const uint32_t b0 = a0 + C::A_BYTES;
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            mma_bf16_lanemask(d, sw128_kmajor_desc(a0 + kk * 32),
                                              sw128_kmajor_desc(b0 + kk * 32), C::IDESC, l0, l1, l2,
                                              l3, 1u);
                        mma_commit(&empty[stage]);
                        if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                    }
                }
                if (!ok) { *s_abort = 1; break; }
                mma_commit(&tfull[acc]);
                mbar_arrive(&mempty[b]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
                if (++b == 2) { b = 0; bphase ^= 1u; }
            }
            mma_commit(final_bar);
            mbar_wait(final_bar, 0, args.status);
        }
        __syncwarp();
    } else {
        // ===================== epilogue (warps 3..6) =====================
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t z[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) z[q] = 0u;
        for (int i = blockIdx.x; i < n_items && !*s_abort; i += gridDim.x) {
            const KUnit u = k_unit(i, n_tiles, args);
            const int sp = u.sp, nt = u.nt;
            const int t = u.mt * BM + row;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(&tfull[acc], acc_phase, args.status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) { *s_abort = 1; break; }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
            uint16_t *dst = args.out + static_cast<size_t>(t) * args.N + nt * BN;
#pragma unroll 1
            for (int cb = 0; cb < BN; cb += 32) {
                uint32_t yr[32];
                tmem_ld32(taddr + cb, yr);
                tmem_ld_wait();
                tmem_st32(taddr + cb, z);
                if (u.slot >= 0) {
                    // fp32 partial of this tail share, compact [slot][BM][BN]
                    if (t < T) {
                        float *pdst = args.tail_partial + (static_cast<size_t>(u.slot) * BM + row) * BN + cb;
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            *reinterpret_cast<float4 *>(pdst + 4 * q) =
                                make_float4(__uint_as_float(yr[4 * q]), __uint_as_float(yr[4 * q + 1]),
                                            __uint_as_float(yr[4 * q + 2]), __uint_as_float(yr[4 * q + 3]));
                    }
                } else if (partial_out) {
                    // fp32 partial of this split; rows past T (and the lanes
                    // the token box did not fill) were masked off and are not stored
                    if (t < T) {
                        float *pdst = args.partial + (static_cast<size_t>(sp) * T + t) * args.N + nt * BN + cb;
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            *reinterpret_cast<float4 *>(pdst + 4 * q) =
                                make_float4(__uint_as_float(yr[4 * q]), __uint_as_float(yr[4 * q + 1]),
                                            __uint_as_float(yr[4 * q + 2]), __uint_as_float(yr[4 * q + 3]));
                    }
                } else if (t < T) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        st_global_cs_v4(dst + cb + 8 * q,
                                     pack_bf16x2(__uint_as_float(yr[8 * q + 0]), __uint_as_float(yr[8 * q + 1])),
                                     pack_bf16x2(__uint_as_float(yr[8 * q + 2]), __uint_as_float(yr[8 * q + 3])),
                                     pack_bf16x2(__uint_as_float(yr[8 * q + 4]), __uint_as_float(yr[8 * q + 5])),
                                     pack_bf16x2(__uint_as_float(yr[8 * q + 6]), __uint_as_float(yr[8 * q + 7])));
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int BN, int AR>
cudaError_t launch_t(const CUtensorMap &tmA, const CUtensorMap &tmB, const KArgs &a, int num_sms,
                     cudaStream_t s, bool dependent = false) {
    using C = KCfg<BN, AR>;
    auto kern = gemm_k_kernel<BN, AR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int m_tiles = (a.T + BM - 1) / BM;
    const int items = k_units(m_tiles, a.N / BN, a);
    const int grid = items < num_sms ? items : num_sms;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = dependent ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, a);
}


// Tail finalize: Y of tail item j (item n_direct + j) is the sum of its nsp
// shares' fp32 partials, added in share order; 8 columns per thread.
constexpr int kFinThreads = 256;

__global__ void __launch_bounds__(kFinThreads)
    gemm_k_tail_finalize_kernel(const float *__restrict__ tp, int n_direct, int tail_items, int nsp,
                                int n_tiles, int bn, int T, int N, uint16_t *__restrict__ out) {
    griddep_wait();  // the partials are the GEMM-K kernel's output
    const int per_item = BM * (bn / 8);
    const long long idx = static_cast<long long>(blockIdx.x) * kFinThreads + threadIdx.x;
    if (idx >= static_cast<long long>(tail_items) * per_item) return;
    const int j = static_cast<int>(idx / per_item);
    const int rem = static_cast<int>(idx - static_cast<long long>(j) * per_item);
    const int r = rem / (bn / 8), c = (rem - r * (bn / 8)) * 8;
    const int item = n_direct + j;
    const int mt = item / n_tiles, nt = item - mt * n_tiles;
    const int t = mt * BM + r;
    if (t >= T) return;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int sp = 0; sp < nsp; ++sp) {
        const float4 *src = reinterpret_cast<const float4 *>(
            tp + (static_cast<size_t>(j * nsp + sp) * BM + r) * bn + c);
        const float4 v0 = src[0], v1 = src[1];
        acc[0] += v0.x; acc[1] += v0.y; acc[2] += v0.z; acc[3] += v0.w;
        acc[4] += v1.x; acc[5] += v1.y; acc[6] += v1.z; acc[7] += v1.w;
    }
    st_global_v4(out + static_cast<size_t>(t) * N + nt * bn + c, pack_bf16x2(acc[0], acc[1]),
                 pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
}

// The tail split: with `items` output tiles on num_sms persistent CTAs, the
// last wave holds items % num_sms tiles.  When that wave would leave at least
// half of the SMs idle, its tiles are cut into s equal shares of their live
// groups (s <= 4, s tiles' shares at most one wave), so the wave takes about
// 1/s of a tile's time.  n_direct < 0: no split.
struct KTailPlan {
    int n_direct, splits;
    size_t bytes;
};

KTailPlan tail_plan(int T, int K, int N, int G, int num_sms) {
    const KTailPlan none{-1, 1, 0};
    const int bn = N % 256 == 0 ? 256 : N % 128 == 0 ? 128 : 64;
    if (T <= 16 || N % bn != 0 || num_sms < 2) return none;
    const long long items = static_cast<long long>((T + BM - 1) / BM) * (N / bn);
    if (items < num_sms || items > (1ll << 30)) return none;
    const int tail = static_cast<int>(items % num_sms);
    if (tail == 0 || 2 * tail > num_sms) return none;
    int s = num_sms / tail;
    s = s > 4 ? 4 : s;
    s = s > K / G ? K / G : s;
    if (s < 2) return none;
    return KTailPlan{static_cast<int>(items - tail), s,
                     static_cast<size_t>(tail) * s * BM * bn * sizeof(float)};
}

}  // namespace

int gemm_k_max_groups() { return kMaxKGroups; }

// Split count (decode, and prefill grids too small for the SMs): each
// 128-column output tile becomes `splits` work items,
// each holding an equal share of the tile's live groups.  The count minimises
// the weight bytes of the busiest CTA (items dealt round-robin over the grid,
// all groups taken as live) plus each SM's share of the fp32 partial traffic
// (written here, read back by the finalize kernel); ties go to fewer splits.
static int split_count(int T, int K, int N, int G, int num_sms, int bn) {
    const int ng = K / G;
    const int n_tiles = N / bn;
    const int m_tiles = T <= 16 ? 1 : (T + BM - 1) / BM;
    double best = 0.0;
    int best_s = 1;
    for (int s = 1; s <= ng; ++s) {
        const int g = (ng + s - 1) / s;
        if ((ng + g - 1) / g != s) continue;  // same shares as a smaller split count
        const long long items = static_cast<long long>(m_tiles) * n_tiles * s;
        const long long waves = (items + num_sms - 1) / num_sms;
        const double cta_bytes = static_cast<double>(waves) * g * G * bn * 2;
        const double partial = s > 1 ? static_cast<double>(s) * T * N * 8 / num_sms : 0.0;
        const double cost = cta_bytes + partial;
        if (s == 1 || cost < best) {
            best = cost;
            best_s = s;
        }
    }
    return best_s;
}

// Decode output tiles: 256 columns when N allows.  Each item then streams a
// weight tile twice as wide per staged token block, and the items are fewer
// (8B down on 152 SMs: 16 tiles x 19 splits = 304 items in two waves, against
// 32 x 14 = 448 in three with 128-column tiles); measured 2-4 us faster per
// decode FFN step at T = 1..16.
int gemm_k_decode_bn(int N) { return N % 256 == 0 ? 256 : 128; }

int gemm_k_decode_splits(int T, int K, int N, int G, int num_sms) {
    return split_count(T, K, N, G, num_sms, gemm_k_decode_bn(N));
}

int gemm_k_split_bn(int N) { return N % 256 == 0 ? 256 : 128; }

int gemm_k_prefill_splits(int T, int K, int N, int G, int num_sms) {
    if (T <= 16 || N % 128 != 0) return 1;
    // splitting only pays while the unsplit grid leaves SMs idle: past that,
    // every split adds partial traffic and item overhead to the same MMA work
    const long long items = static_cast<long long>((T + BM - 1) / BM) * (N / gemm_k_split_bn(N));
    if (items >= num_sms) return 1;
    return split_count(T, K, N, G, num_sms, gemm_k_split_bn(N));
}

size_t gemm_k_split_workspace_bytes(int T, int K, int N, int G, int num_sms) {
    const int s = gemm_k_prefill_splits(T, K, N, G, num_sms);
    return s > 1 ? static_cast<size_t>(s) * T * N * sizeof(float) : 0;
}

cudaError_t launch_gemm_k_split(const CUtensorMap &tmA, const CUtensorMap &tmB, const KArgs &a0,
                                float *ws, int num_sms, cudaStream_t s) {
    KArgs a = a0;
    a.splits = gemm_k_prefill_splits(a.T, a.K, a.N, a.G, num_sms);
    a.partial = ws;
    cudaError_t e = gemm_k_split_bn(a.N) == 256 ? launch_t<256, BM>(tmA, tmB, a, num_sms, s)
                                                : launch_t<128, BM>(tmA, tmB, a, num_sms, s);
    if (e != cudaSuccess) return e;
    return launch_decode_k_finalize(ws, a.splits, a.T * a.N, a.out, s);
}

size_t gemm_k_decode_workspace_bytes(int T, int K, int N, int G, int num_sms) {
    return static_cast<size_t>(gemm_k_decode_splits(T, K, N, G, num_sms)) * T * N * sizeof(float);
}

cudaError_t launch_gemm_k_decode(const CUtensorMap &tmA, const CUtensorMap &tmB, const KArgs &a0,
                                 float *ws, int num_sms, cudaStream_t s) {
    KArgs a = a0;
    a.splits = gemm_k_decode_splits(a.T, a.K, a.N, a.G, num_sms);
    a.partial = ws;
    // a programmatic dependent of the kernel before it (the decode gate/up)
    cudaError_t e = gemm_k_decode_bn(a.N) == 256 ? launch_t<256, 16>(tmA, tmB, a, num_sms, s, true)
                                                 : launch_t<128, 16>(tmA, tmB, a, num_sms, s, true);
    if (e != cudaSuccess) return e;
    return launch_decode_k_finalize(ws, a.splits, a.T * a.N, a.out, s);
}

size_t gemm_k_tail_workspace_bytes(int T, int K, int N, int G, int num_sms) {
    return tail_plan(T, K, N, G, num_sms).bytes;
}

cudaError_t launch_gemm_k_tail(int bn, const CUtensorMap &tmA, const CUtensorMap &tmB, const KArgs &a0,
                               float *ws, int num_sms, cudaStream_t s) {
    const KTailPlan p = tail_plan(a0.T, a0.K, a0.N, a0.G, num_sms);
    const int expect_bn = a0.N % 256 == 0 ? 256 : a0.N % 128 == 0 ? 128 : 64;
    if (p.n_direct < 0 || bn != expect_bn || ws == nullptr) return cudaErrorInvalidValue;
    KArgs a = a0;
    a.splits = 1;
    a.partial = nullptr;
    a.n_direct = p.n_direct;
    a.tail_splits = p.splits;
    a.tail_partial = ws;
    cudaError_t e = launch_gemm_k(bn, tmA, tmB, a, num_sms, s);
    if (e != cudaSuccess) return e;
    const int n_tiles = a.N / bn;
    const int tail_items = ((a.T + BM - 1) / BM) * n_tiles - p.n_direct;
    const long long threads = static_cast<long long>(tail_items) * BM * (bn / 8);
    // a programmatic dependent of the GEMM-K kernel: its launch overlaps that
    // kernel's tail, and griddep_wait orders its reads after the partials
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((threads + kFinThreads - 1) / kFinThreads));
    cfg.blockDim = dim3(kFinThreads);
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_k_tail_finalize_kernel, static_cast<const float *>(ws), p.n_direct,
                              tail_items, p.splits, n_tiles, bn, a.T, a.N, a.out);
}

cudaError_t launch_gemm_k(int bn, const CUtensorMap &tmA, const CUtensorMap &tmB, const KArgs &a,
                          int num_sms, cudaStream_t s) {
    if (bn == 256) return launch_t<256, BM>(tmA, tmB, a, num_sms, s);
    if (bn == 128) return launch_t<128, BM>(tmA, tmB, a, num_sms, s);
    if (bn == 64) return launch_t<64, BM>(tmA, tmB, a, num_sms, s);
    return cudaErrorInvalidValue;
}

}  // namespace wide
