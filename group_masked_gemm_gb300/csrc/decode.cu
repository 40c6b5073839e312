// decode.cu -- small-T (decode) group-masked projections (WIDE, App. B:
// GEMV variants of GEMM-MN and GEMM-K; for decoding the mask reordering is
// bypassed and routing is checked directly at block level).
//
// With at most 16 tokens the work is bound by HBM reads of the weights, so
// the kernels read only the weight groups that at least one token uses (the
// union of the tokens' active groups), with 16-byte non-allocating loads
// issued a whole chunk at a time (8 x 512 B per warp and weight row) so that
// enough bytes are in flight to cover the HBM latency.
//   decode_mn:  one warp per output feature n (gate and up rows together),
//               X staged once per persistent CTA in shared memory.
//   decode_k :  the reduction dimension is split, on group boundaries, over
//               gridDim.y CTAs; each CTA stages its slice of the token rows
//               (inactive groups zeroed) once, streams 16 output rows of W
//               and writes fp32 partial sums to the workspace; a second
//               kernel adds the partials of each output in split order
//               (deterministic) and rounds to bf16.
#include "common.cuh"
#include "internal.h"

namespace wide {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kChunkIters = 8;      // 256-element steps whose loads are issued together
constexpr int kSliceBytes = 96 * 1024;  // staged token-row slice of one decode_k CTA

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

// Per-group bitmask of active tokens (bit t set when M[t, g] != 0), groups [g0, g1).
__device__ __forceinline__ void build_group_bits(const uint8_t *mask, int T, int ng, int g0,
                                                 int g1, uint32_t *gbits) {
    for (int g = g0 + static_cast<int>(threadIdx.x); g < g1; g += blockDim.x) {
        uint32_t b = 0;
        for (int t = 0; t < T; ++t) b |= static_cast<uint32_t>(mask[t * ng + g] != 0) << t;
        gbits[g - g0] = b;
    }
}

template <MNMode MODE, int TM>
__global__ void __launch_bounds__(kThreads)
    decode_mn_kernel(const DecodeArgs a) {
    // a kernel launched after this one as a programmatic dependent (the decode
    // GEMM-K) may set itself up now; it waits for this grid before any input
    griddep_launch_dependents();
    extern __shared__ __align__(16) uint8_t smem[];
    const int T = a.T, K = a.K, N = a.N, G = a.G;
    const int ng = N / G;
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem);                      // [T][K]
    uint32_t *gbits = reinterpret_cast<uint32_t *>(smem + static_cast<size_t>(TM) * K * 2);  // [ng]
    int *glist = reinterpret_cast<int *>(gbits + ng);                                          // [ng]
    __shared__ int s_live;

    for (int v = threadIdx.x; v < T * K / 8; v += kThreads)
        reinterpret_cast<uint4 *>(xs)[v] = reinterpret_cast<const uint4 *>(a.x)[v];
    build_group_bits(a.mask, T, ng, 0, ng, gbits);
    __syncthreads();
    if (threadIdx.x == 0) {  // groups some token uses, ascending
        int c = 0;
        for (int g = 0; g < ng; ++g)
            if (gbits[g] != 0u) glist[c++] = g;
        s_live = c;
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_warps = gridDim.x * kWarps;
    const int gw = blockIdx.x * kWarps + warp;
    // rows of groups no token uses: zeros, without reading their weights
    for (int n = gw; n < N; n += n_warps)
        if (gbits[n / G] == 0u && lane < T) a.out[static_cast<size_t>(lane) * N + n] = 0;
    // rows of the live groups, dealt evenly over all warps of the grid
    const int n_active = s_live * G;
    for (int ia = gw; ia < n_active; ia += n_warps) {
        const int n = glist[ia / G] * G + ia % G;
        const uint32_t bits = gbits[n / G];
        float acc0[TM], acc1[TM];
#pragma unroll
        for (int t = 0; t < TM; ++t) acc0[t] = acc1[t] = 0.f;
        const uint16_t *w0 = a.w0 + static_cast<size_t>(n) * K;
        const uint16_t *w1 = MODE == MNMode::kGateUp ? a.w1 + static_cast<size_t>(n) * K : nullptr;
        for (int kc = 0; kc < K; kc += 256 * kChunkIters) {
            uint4 r0[kChunkIters], r1[kChunkIters];
#pragma unroll
            for (int j = 0; j < kChunkIters; ++j) {
                const int k = kc + 256 * j + lane * 8;
                if (k < K) {
                    r0[j] = ld_stream16(w0 + k);
                    if (MODE == MNMode::kGateUp) r1[j] = ld_stream16(w1 + k);
                }
            }
#pragma unroll
            for (int j = 0; j < kChunkIters; ++j) {
                const int k = kc + 256 * j + lane * 8;
                if (k >= K) break;
                float f0[8], f1[8];
                bf16x8_to_f32(r0[j], f0);
                if (MODE == MNMode::kGateUp) bf16x8_to_f32(r1[j], f1);
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

// Partial sums of one split (blockIdx.y) of the reduction dimension for 16
// output rows: ws[split][t][n] (fp32).
template <int TM>
__global__ void __launch_bounds__(kThreads)
    decode_k_partial_kernel(const DecodeArgs a, int groups_per_split, float *ws) {
    griddep_launch_dependents();  // see launch_decode_k_finalize
    extern __shared__ __align__(16) uint8_t smem[];
    const int T = a.T, K = a.K, N = a.N, G = a.G;
    const int ng = K / G;
    const int g_begin = blockIdx.y * groups_per_split;
    const int g_end = min(ng, g_begin + groups_per_split);
    const int k0 = g_begin * G;
    const int klen = (g_end - g_begin) * G;
    const int kstride = groups_per_split * G;  // row stride of the staged slice
    uint16_t *as = reinterpret_cast<uint16_t *>(smem);                                  // [TM][kstride]
    uint32_t *gbits = reinterpret_cast<uint32_t *>(smem + static_cast<size_t>(TM) * kstride * 2);

    build_group_bits(a.mask, T, ng, g_begin, g_end, gbits);
    __syncthreads();
    const int vec_per_row = klen / 8;
    for (int v = threadIdx.x; v < T * vec_per_row; v += kThreads) {
        const int t = v / vec_per_row, k = (v - t * vec_per_row) * 8;
        uint4 val = make_uint4(0, 0, 0, 0);
        if ((gbits[k / G] >> t) & 1u)
            val = *reinterpret_cast<const uint4 *>(a.x + static_cast<size_t>(t) * K + k0 + k);
        *reinterpret_cast<uint4 *>(as + t * kstride + k) = val;
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kRowsPerCta + warp * kRowsPerWarp;
    float acc[kRowsPerWarp][TM];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int t = 0; t < TM; ++t) acc[r][t] = 0.f;

    for (int kc = 0; kc < klen; kc += 256 * kChunkIters) {
        uint4 wr[kChunkIters][kRowsPerWarp];
#pragma unroll
        for (int j = 0; j < kChunkIters; ++j) {
            const int k = kc + 256 * j + lane * 8;
            // a group no token uses is never read
            if (k < klen && gbits[k / G] != 0u) {
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r)
                    wr[j][r] = ld_stream16(a.w0 + static_cast<size_t>(n0 + r) * K + k0 + k);
            }
        }
#pragma unroll
        for (int j = 0; j < kChunkIters; ++j) {
            const int k = kc + 256 * j + lane * 8;
            if (k >= klen) break;
            const uint32_t bits = gbits[k / G];
            if (bits == 0u) continue;
            float w[kRowsPerWarp][8];
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) bf16x8_to_f32(wr[j][r], w[r]);
#pragma unroll
            for (int t = 0; t < TM; ++t) {
                if (t < T && ((bits >> t) & 1u)) {
                    float xf[8];
                    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(as + t * kstride + k), xf);
#pragma unroll
                    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[r][t] = fmaf(w[r][e], xf[e], acc[r][t]);
                }
            }
        }
    }
    float *out = ws + static_cast<size_t>(blockIdx.y) * T * N;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int t = 0; t < TM; ++t) {
            if (t >= T) break;
            const float s = warp_sum(acc[r][t]);
            if (lane == 0) out[static_cast<size_t>(t) * N + n0 + r] = s;
        }
}

// Y[t][n] = bf16( sum over splits s = 0, 1, ... of ws[s][t][n] ).
__global__ void __launch_bounds__(kThreads)
    decode_k_finalize_kernel(const float *ws, int splits, int TN, uint16_t *out) {
    griddep_wait();  // the partials are the previous kernel's output
    const int i = blockIdx.x * kThreads + threadIdx.x;
    if (i >= TN) return;
    float s = 0.f;
    for (int p = 0; p < splits; ++p) s += ws[static_cast<size_t>(p) * TN + i];
    out[i] = f32_to_bf16_bits(s);
}

template <MNMode MODE, int TM>
cudaError_t launch_mn_t(const DecodeArgs &a, int num_sms, cudaStream_t s) {
    auto kern = decode_mn_kernel<MODE, TM>;
    const size_t smem = decode_mn_smem_bytes(a.T, a.K, a.N / a.G);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int rows_blocks = (a.N + kWarps - 1) / kWarps;
    const int per_sm = smem <= 100 * 1024 ? 2 : 1;  // more CTAs per SM measured slower (prologue per CTA)
    const int grid = rows_blocks < per_sm * num_sms ? rows_blocks : per_sm * num_sms;
    kern<<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

int tm_of(int T) { return T <= 1 ? 1 : T <= 4 ? 4 : 16; }

}  // namespace

size_t decode_mn_smem_bytes(int T, int K, int n_groups) {
    return static_cast<size_t>(tm_of(T)) * K * 2 + static_cast<size_t>(n_groups) * 8;  // X rows, group bits, live list
}

// Groups per split of the reduction dimension: the staged slice of TM token
// rows fits kSliceBytes.
int decode_k_groups_per_split(int T, int K, int G) {
    const int ng = K / G;
    int gps_max = kSliceBytes / (tm_of(T) * G * 2);
    if (gps_max < 1) gps_max = 1;
    const int splits = (ng + gps_max - 1) / gps_max;
    return (ng + splits - 1) / splits;  // equal splits on group boundaries
}

size_t decode_k_smem_bytes(int T, int K, int G) {
    const int gps = decode_k_groups_per_split(T, K, G);
    return static_cast<size_t>(tm_of(T)) * gps * G * 2 + static_cast<size_t>(gps) * 4;
}

size_t decode_k_workspace_bytes(int T, int K, int N, int G) {
    const int ng = K / G;
    const int gps = decode_k_groups_per_split(T, K, G);
    const int splits = (ng + gps - 1) / gps;
    return static_cast<size_t>(splits) * T * N * sizeof(float);
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

template <int TM>
static cudaError_t launch_k_partial(const DecodeArgs &a, int gps, int splits, float *ws,
                                    cudaStream_t s) {
    auto kern = decode_k_partial_kernel<TM>;
    const size_t smem = static_cast<size_t>(TM) * gps * a.G * 2 + static_cast<size_t>(gps) * 4;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<dim3(a.N / kRowsPerCta, splits), kThreads, smem, s>>>(a, gps, ws);
    return cudaGetLastError();
}

// The finalize is launched as a programmatic dependent of the partial-sum
// kernel before it (which triggers early): its launch overlaps that kernel,
// and griddep_wait holds it until the partials are complete and visible.
cudaError_t launch_decode_k_finalize(const float *ws, int splits, int TN, uint16_t *out,
                                     cudaStream_t s) {
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((TN + kThreads - 1) / kThreads);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_k_finalize_kernel, ws, splits, TN, out);
}

cudaError_t launch_decode_k(const DecodeArgs &a, float *ws, cudaStream_t s) {
    const int ng = a.K / a.G;
    const int gps = decode_k_groups_per_split(a.T, a.K, a.G);
    const int splits = (ng + gps - 1) / gps;
    cudaError_t e;
    if (a.T <= 1) e = launch_k_partial<1>(a, gps, splits, ws, s);
    else if (a.T <= 4) e = launch_k_partial<4>(a, gps, splits, ws, s);
    else e = launch_k_partial<16>(a, gps, splits, ws, s);
    if (e != cudaSuccess) return e;
    return launch_decode_k_finalize(ws, splits, a.T * a.N, a.out, s);
}

}  // namespace wide

// ---------------------------------------------------------------------------
// Allocation-free decode GEMM-K.
//
// Some callers of this library cannot allocate device memory: code running
// under a memory planner that owns every device allocation, plugin hosts that
// hand a kernel no workspace, or paths where a cudaMalloc (which can
// synchronise the device) is not acceptable.  For them the decode GEMM-K
// keeps its fp32 partial sums in this fixed array instead of a caller
// workspace.  It is part of the module, so every GPU that loads the library
// holds it until the process exits.
#include <mutex>

#include "../../include/wide.h"

namespace {

constexpr size_t kStaticScratchBytes = WIDE_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) float g_static_scratch[kStaticScratchBytes / sizeof(float)];

constexpr int kMaxStaticDevices = 64;
std::mutex g_static_mutex;
float *g_static_scratch_ptr[kMaxStaticDevices] = {nullptr};
int g_static_num_sms[kMaxStaticDevices] = {0};

// Device address of g_static_scratch on the current device.  The first call
// on each device looks it up (cudaGetSymbolAddress) and caches it.
wide_status_t static_scratch_for_current_device(float **ptr, int *num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxStaticDevices)
        return WIDE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (g_static_scratch_ptr[dev] == nullptr) {
        float *p = nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_static_scratch) != cudaSuccess ||
            p == nullptr)
            return WIDE_ERR_CUDA;
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return WIDE_ERR_CUDA;
        g_static_scratch_ptr[dev] = p;
        g_static_num_sms[dev] = n;
    }
    *ptr = g_static_scratch_ptr[dev];
    *num_sms = g_static_num_sms[dev];
    return WIDE_OK;
}

bool aligned16_ptr(const void *p) {
    return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

}  // namespace

extern "C" wide_status_t wide_gemm_k_decode_noalloc(const uint16_t *A, const uint16_t *W,
                                                    const uint8_t *mask, int T, int K, int N,
                                                    int G, uint16_t *Y, void *stream) {
    if (!aligned16_ptr(A) || !aligned16_ptr(W) || !aligned16_ptr(mask) || !aligned16_ptr(Y))
        return WIDE_ERR_INVALID_ARG;
    if (T < 1 || T > 16 || K < 64 || N < 64 || K % 64 || N % 64) return WIDE_ERR_INVALID_ARG;
    if (!(G == 64 || G == 128 || G == 256 || G == 512))
        return (G >= 16 && (G & (G - 1)) == 0) ? WIDE_ERR_UNSUPPORTED : WIDE_ERR_INVALID_ARG;
    if (K % G) return WIDE_ERR_INVALID_ARG;
    if (wide::decode_k_workspace_bytes(T, K, N, G) > kStaticScratchBytes) return WIDE_ERR_WORKSPACE;
    float *scratch = nullptr;
    int num_sms = 0;
    wide_status_t st = static_scratch_for_current_device(&scratch, &num_sms);
    if (st != WIDE_OK) return st;
    (void)num_sms;
    wide::DecodeArgs a{A, W, nullptr, mask, Y, T, K, N, G};
    return wide::launch_decode_k(a, scratch, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? WIDE_OK
               : WIDE_ERR_CUDA;
}
