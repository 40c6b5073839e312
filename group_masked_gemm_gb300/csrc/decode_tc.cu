// decode_tc.cu -- small-T (decode) GEMM-MN on tcgen05 (WIDE, App. B: GEMV
// variant of GEMM-MN; in decoding the mask reordering is bypassed and routing
// is checked at block level).
//
// Decode is bound by HBM reads of the weight groups some token uses.  The
// products are computed transposed, D[row, token] = sum_k W[row,k] X[token,k],
// so the weight rows are the M = 128 side of the MMA -- streamed by TMA,
// 6 stages deep -- and the <= 16 tokens are the N = 16 side (rows past T are
// zero).  The tensor core keeps the per-byte arithmetic (16 MACs per weight
// element at T = 16) off the CUDA cores.
//   decode_mn_tc: one CTA per (group, 32-row slice).  Groups no token uses
//                 write zeros and never read their weights.  For gate/up the
//                 A tile holds the 32 gate rows in rows 0..31 and the 32 up
//                 rows in rows 64..95, so one MMA computes both.
// It serves 5 <= T <= 16; smaller batches go to the CUDA-core kernel of
// decode.cu, which streams the same bytes with less issue overhead.
#include "common.cuh"
#include "internal.h"

namespace wide {
namespace {

constexpr int kTcThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int BK = 64;
constexpr int NTOK = 16;
constexpr int A_BYTES = 128 * BK * 2;     // weight tile, M = 128 rows
constexpr int XB_BYTES = NTOK * BK * 2;   // token tile, N = 16 rows
constexpr uint32_t IDESC = idesc_bf16_f32(128, NTOK);
constexpr int TMEM_COLS = 32;
constexpr int RT = 32;                    // weight rows per decode_mn_tc CTA (per weight)

constexpr int MN_STAGES = 5;
constexpr int MN_STAGE_BYTES = A_BYTES + XB_BYTES;
constexpr int SCRATCH_BYTES = 128 * (NTOK + 1) * 4;
// TMEM: two fp32 accumulators of NTOK columns (double-buffered across items)
constexpr int MN_SMEM = 1024 + MN_STAGES * MN_STAGE_BYTES + SCRATCH_BYTES + 256;
static_assert(2 * MN_SMEM <= 227 * 1024, "two decode_mn_tc CTAs per SM");

__device__ __forceinline__ uint16_t to_bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&h);
}

// Tokens of the decode batch active in group g (bit t), computed by one warp.
__device__ __forceinline__ uint32_t group_token_bits(const uint8_t *mask, int T, int ng, int g) {
    const int lane = threadIdx.x & 31;
    return __ballot_sync(0xffffffffu, lane < T && mask[lane * ng + g] != 0);
}

template <MNMode MODE>
__global__ void __launch_bounds__(kTcThreads)
    decode_mn_tc_kernel(const __grid_constant__ CUtensorMap tmW0,
                        const __grid_constant__ CUtensorMap tmW1,
                        const __grid_constant__ CUtensorMap tmX, const DecodeArgs a, int *status) {
    griddep_launch_dependents();  // see decode_mn_kernel
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float *scratch = reinterpret_cast<float *>(smem + MN_STAGES * MN_STAGE_BYTES);  // [128][17]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + MN_STAGES * MN_STAGE_BYTES + SCRATCH_BYTES);
    uint64_t *full = bars, *empty = bars + MN_STAGES;
    uint64_t *tfull = bars + 2 * MN_STAGES, *tempty = tfull + 2;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(tempty + 2);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = a.T, K = a.K, N = a.N, G = a.G;
    const int ng = N / G;
    const int n_sub = G / RT;
    const int n_items = ng * n_sub;

    if (threadIdx.x == 0) {
        for (int s = 0; s < MN_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);
        }
        *s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmW0);
        if (MODE == MNMode::kGateUp) prefetch_tmap(&tmW1);
        prefetch_tmap(&tmX);
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const int k_blocks = K / BK;
    // the token box has min(T, 16) rows; rows T..15 of the tile keep stale data
    // and only feed output columns t >= T, which are never stored
    const uint32_t kBytes = (MODE == MNMode::kGateUp ? 2 : 1) * RT * BK * 2 + min(T, NTOK) * BK * 2;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        int stage = 0;
        uint32_t phase = 0, used = 0, last_parity = 0;
        for (int i = blockIdx.x; i < n_items && !*s_abort; i += gridDim.x) {
            const int g = i / n_sub;
            if (group_token_bits(a.mask, T, ng, g) == 0u) continue;  // weights never read
            const int row0 = g * G + (i - g * n_sub) * RT;
            for (int kb = 0; kb < k_blocks; ++kb) {
                int ok = 1;
                if (lane == 0) ok = mbar_wait(&empty[stage], phase ^ 1u, status);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) { *s_abort = 1; break; }
                if (lane == 0) {
                    uint8_t *st = smem + stage * MN_STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[stage], kBytes);
                    tma_load_2d(st, &tmW0, &full[stage], kb * BK, row0);
                    if (MODE == MNMode::kGateUp)
                        tma_load_2d(st + 64 * 128, &tmW1, &full[stage], kb * BK, row0);
                    tma_load_2d(st + A_BYTES, &tmX, &full[stage], kb * BK, 0);
                }
                used |= 1u << stage;
                last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == MN_STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (lane == 0)
            for (int s = 0; s < MN_STAGES; ++s)
                if (used & (1u << s)) mbar_wait(&full[s], (last_parity >> s) & 1u, status);
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        int stage = 0, acc = 0;
        uint32_t phase = 0, acc_phase = 0;
        for (int i = blockIdx.x; i < n_items && !*s_abort; i += gridDim.x) {
            const int g = i / n_sub;
            if (group_token_bits(a.mask, T, ng, g) == 0u) continue;
            if (lane == 0) {
                bool ok = mbar_wait(&tempty[acc], acc_phase ^ 1u, status);
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * NTOK);
                for (int kb = 0; kb < k_blocks && ok; ++kb) {
                    if (!mbar_wait(&full[stage], phase, status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(smem + stage * MN_STAGE_BYTES);
                    const uint32_t x0 = a0 + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_bf16(d, sw128_kmajor_desc(a0 + kk * 32), sw128_kmajor_desc(x0 + kk * 32),
                                 IDESC, (kb | kk) != 0);
                    mma_commit(&empty[stage]);
                    if (++stage == MN_STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) *s_abort = 1;
                else mma_commit(&tfull[acc]);
            }
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            __syncwarp();
        }
        if (lane == 0) {
            mma_commit(&tfull[acc]);  // drains every MMA issued so far
            mbar_wait(&tfull[acc], acc_phase, status);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int i = blockIdx.x; i < n_items && !*s_abort; i += gridDim.x) {
            const int g = i / n_sub;
            const int row0 = g * G + (i - g * n_sub) * RT;
            const uint32_t bits = group_token_bits(a.mask, T, ng, g);
            if (bits == 0u) {  // no token uses this group: zeros
                for (int j = threadIdx.x - 64; j < T * RT; j += 128)
                    a.out[static_cast<size_t>(j / RT) * N + row0 + j % RT] = 0;
                continue;
            }
            int ok = 1;
            if (lane == 0) ok = mbar_wait(&tfull[acc], acc_phase, status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) { *s_abort = 1; break; }
            tc_fence_after();
            uint32_t v[16];
            tmem_ld16(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * NTOK, v);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
#pragma unroll
            for (int t = 0; t < NTOK; ++t) scratch[r * (NTOK + 1) + t] = __uint_as_float(v[t]);
            named_barrier_sync(1, 128);
            for (int j = threadIdx.x - 64; j < T * RT; j += 128) {
                const int t = j / RT, rr = j - t * RT;
                float y = 0.f;
                if ((bits >> t) & 1u) {
                    const float g0 = scratch[rr * (NTOK + 1) + t];
                    if (MODE == MNMode::kGateUp) {
                        const float u = scratch[(64 + rr) * (NTOK + 1) + t];
                        y = __fdividef(g0, 1.0f + __expf(-g0)) * u;
                    } else {
                        y = g0;
                    }
                }
                a.out[static_cast<size_t>(t) * N + row0 + rr] = to_bf16_bits(y);
            }
            named_barrier_sync(1, 128);  // scratch is reused by the next item
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <MNMode MODE>
cudaError_t launch_mn(const CUtensorMap &tmW0, const CUtensorMap &tmW1, const CUtensorMap &tmX,
                      const DecodeArgs &a, int *status, int num_sms, cudaStream_t s) {
    auto kern = decode_mn_tc_kernel<MODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, MN_SMEM);
    if (e != cudaSuccess) return e;
    const int items = (a.N / a.G) * (a.G / RT);
    const int grid = items < 2 * num_sms ? items : 2 * num_sms;  // two CTAs per SM
    kern<<<grid, kTcThreads, MN_SMEM, s>>>(tmW0, tmW1, tmX, a, status);
    return cudaGetLastError();
}

}  // namespace

int decode_tc_rows_per_item() { return RT; }

cudaError_t launch_decode_mn_tc(MNMode mode, const CUtensorMap &tmW0, const CUtensorMap &tmW1,
                                const CUtensorMap &tmX, const DecodeArgs &a, int *status,
                                int num_sms, cudaStream_t s) {
    if (mode == MNMode::kGateUp)
        return launch_mn<MNMode::kGateUp>(tmW0, tmW1, tmX, a, status, num_sms, s);
    return launch_mn<MNMode::kPlain>(tmW0, tmW1, tmX, a, status, num_sms, s);
}

}  // namespace wide
