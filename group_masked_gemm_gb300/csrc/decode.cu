// decode.cu -- small-T (decode) group-masked projections (WIDE, App. B:
// GEMV variants of GEMM-MN and GEMM-K; for decoding the mask reordering is
// bypassed and routing is checked directly at block level).
//
// With at most 16 tokens the work is bound by HBM reads of the weights, so
// the kernels stream only the weight groups that at least one token uses
// (the union of the tokens' active groups) with 16-byte non-allocating loads
// and keep the few token rows on chip.
//   decode_mn: one warp per output feature n (gate and up rows together),
//              X staged once per persistent CTA in shared memory.
//   decode_k : a CTA owns 16 output features; the reduction dimension is
//              walked in chunks whose token rows are staged, already masked
//              (inactive groups zeroed), in shared memory; loads of W[n, K_g]
//              are issued only for groups in the token union.
#include "common.cuh"
#include "internal.h"

namespace wide {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
    return v;
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&h);
}

// Per-group bitmask of active tokens (bit t set when M[t, g] != 0).
__device__ __forceinline__ void build_group_bits(const uint8_t *mask, int T, int ng,
                                                 uint32_t *gbits) {
    for (int g = threadIdx.x; g < ng; g += blockDim.x) {
        uint32_t b = 0;
        for (int t = 0; t < T; ++t) b |= static_cast<uint32_t>(mask[t * ng + g] != 0) << t;
        gbits[g] = b;
    }
}

template <MNMode MODE, int TM>
__global__ void __launch_bounds__(kThreads)
    decode_mn_kernel(const DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int T = a.T, K = a.K, N = a.N, G = a.G;
    const int ng = N / G;
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem);                      // [T][K]
    uint32_t *gbits = reinterpret_cast<uint32_t *>(smem + static_cast<size_t>(TM) * K * 2);

    for (int v = threadIdx.x; v < T * K / 8; v += kThreads)
        reinterpret_cast<uint4 *>(xs)[v] = reinterpret_cast<const uint4 *>(a.x)[v];
    build_group_bits(a.mask, T, ng, gbits);
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_warps = gridDim.x * kWarps;
    for (int n = blockIdx.x * kWarps + warp; n < N; n += n_warps) {
        const uint32_t bits = gbits[n / G];
        if (bits == 0) {
            if (lane < T) a.out[static_cast<size_t>(lane) * N + n] = 0;
            continue;
        }
        float acc0[TM], acc1[TM];
#pragma unroll
        for (int t = 0; t < TM; ++t) acc0[t] = acc1[t] = 0.f;
        const uint16_t *w0 = a.w0 + static_cast<size_t>(n) * K;
        const uint16_t *w1 = MODE == MNMode::kGateUp ? a.w1 + static_cast<size_t>(n) * K : nullptr;
#pragma unroll 4
        for (int k = lane * 8; k < K; k += 256) {
            float f0[8], f1[8];
            bf16x8_to_f32(ld_stream16(w0 + k), f0);
            if (MODE == MNMode::kGateUp) bf16x8_to_f32(ld_stream16(w1 + k), f1);
#pragma unroll
            for (int t = 0; t < TM; ++t) {
                if (t < T && ((bits >> t) & 1u)) {
                    float xf[8];
                    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(xs + t * K + k), xf);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        acc0[t] = fmaf(f0[e], xf[e], acc0[t]);
                        if (MODE == MNMode::kGateUp) acc1[t] = fmaf(f1[e], xf[e], acc1[t]);
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < TM; ++t) {
            if (t >= T) break;
            const float s0 = warp_sum(acc0[t]);
            float r = s0;
            if (MODE == MNMode::kGateUp) {
                const float s1 = warp_sum(acc1[t]);
                r = __fdividef(s0, 1.0f + __expf(-s0)) * s1;
            }
            if (lane == 0)
                a.out[static_cast<size_t>(t) * N + n] = ((bits >> t) & 1u) ? f32_to_bf16_bits(r) : 0;
        }
    }
}

constexpr int kRowsPerWarp = 2;
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;
constexpr int kChunk = 1024;  // reduction columns staged per step

template <int TM>
__global__ void __launch_bounds__(kThreads)
    decode_k_kernel(const DecodeArgs a) {
    __shared__ __align__(16) uint16_t as[TM * kChunk];
    extern __shared__ __align__(16) uint8_t dsmem[];
    uint32_t *gbits = reinterpret_cast<uint32_t *>(dsmem);
    const int T = a.T, K = a.K, N = a.N, G = a.G;
    const int ng = K / G;
    build_group_bits(a.mask, T, ng, gbits);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kRowsPerCta + warp * kRowsPerWarp;
    float acc[kRowsPerWarp][TM];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int t = 0; t < TM; ++t) acc[r][t] = 0.f;

    for (int kc = 0; kc < K; kc += kChunk) {
        const int len = min(kChunk, K - kc);
        __syncthreads();  // previous chunk consumed; gbits ready on the first pass
        for (int v = threadIdx.x; v < T * (len / 8); v += kThreads) {
            const int t = v / (len / 8), k = (v - t * (len / 8)) * 8;
            const bool on = (gbits[(kc + k) / G] >> t) & 1u;
            uint4 val = make_uint4(0, 0, 0, 0);
            if (on) val = *reinterpret_cast<const uint4 *>(a.x + static_cast<size_t>(t) * K + kc + k);
            *reinterpret_cast<uint4 *>(as + t * kChunk + k) = val;
        }
        __syncthreads();
#pragma unroll 2
        for (int k = lane * 8; k < len; k += 256) {
            const uint32_t bits = gbits[(kc + k) / G];
            if (bits == 0) continue;  // no token uses this group: its weights are never read
            float w[kRowsPerWarp][8];
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r)
                bf16x8_to_f32(ld_stream16(a.w0 + static_cast<size_t>(n0 + r) * K + kc + k), w[r]);
#pragma unroll
            for (int t = 0; t < TM; ++t) {
                if (t < T && ((bits >> t) & 1u)) {
                    float xf[8];
                    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(as + t * kChunk + k), xf);
#pragma unroll
                    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[r][t] = fmaf(w[r][e], xf[e], acc[r][t]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int t = 0; t < TM; ++t) {
            if (t >= T) break;
            const float s = warp_sum(acc[r][t]);
            if (lane == 0) a.out[static_cast<size_t>(t) * N + n0 + r] = f32_to_bf16_bits(s);
        }
}

template <MNMode MODE, int TM>
cudaError_t launch_mn_t(const DecodeArgs &a, int num_sms, cudaStream_t s) {
    auto kern = decode_mn_kernel<MODE, TM>;
    const size_t smem = static_cast<size_t>(TM) * a.K * 2 + static_cast<size_t>(a.N / a.G) * 4;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int rows_blocks = (a.N + kWarps - 1) / kWarps;
    const int grid = rows_blocks < 2 * num_sms ? rows_blocks : 2 * num_sms;
    kern<<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <int TM>
cudaError_t launch_k_t(const DecodeArgs &a, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(a.K / a.G) * 4;
    decode_k_kernel<TM><<<a.N / kRowsPerCta, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

size_t decode_mn_smem_bytes(int T, int K, int n_groups) {
    const int tm = T <= 1 ? 1 : T <= 4 ? 4 : 16;
    return static_cast<size_t>(tm) * K * 2 + static_cast<size_t>(n_groups) * 4;
}

cudaError_t launch_decode_mn(MNMode mode, const DecodeArgs &a, int num_sms, cudaStream_t s) {
    if (mode == MNMode::kGateUp) {
        if (a.T <= 1) return launch_mn_t<MNMode::kGateUp, 1>(a, num_sms, s);
        if (a.T <= 4) return launch_mn_t<MNMode::kGateUp, 4>(a, num_sms, s);
        return launch_mn_t<MNMode::kGateUp, 16>(a, num_sms, s);
    }
    if (a.T <= 1) return launch_mn_t<MNMode::kPlain, 1>(a, num_sms, s);
    if (a.T <= 4) return launch_mn_t<MNMode::kPlain, 4>(a, num_sms, s);
    return launch_mn_t<MNMode::kPlain, 16>(a, num_sms, s);
}

cudaError_t launch_decode_k(const DecodeArgs &a, int num_sms, cudaStream_t s) {
    (void)num_sms;
    if (a.T <= 1) return launch_k_t<1>(a, s);
    if (a.T <= 4) return launch_k_t<4>(a, s);
    return launch_k_t<16>(a, s);
}

}  // namespace wide
