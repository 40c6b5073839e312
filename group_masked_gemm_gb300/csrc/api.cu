// api.cu -- the extern "C" boundary of libwide.so (declared in include/wide.h):
// host-side argument validation, TMA descriptor encoding, kernel dispatch
// (prefill tcgen05 kernels vs. small-T decode kernels) and the device status
// word.  No call allocates, frees or synchronises (except wide_device_status).
#include <cudaTypedefs.h>

#include <cstdlib>
#include <mutex>

#include "../../include/wide.h"
#include "common.cuh"
#include "internal.h"
#include "partition.cuh"

namespace wide {
int gemm_k_max_groups();
}  // namespace wide

namespace {

constexpr int kVersion = 1 * 10000 + 0 * 100 + 0;
constexpr int kDecodeMaxT = 16;
constexpr int kMaxDevices = 64;

// First device-side failure since the last wide_device_status() call.
__device__ int g_device_status = 0;

std::mutex g_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
int g_num_sms[kMaxDevices] = {0};
int *g_status_ptr[kMaxDevices] = {nullptr};

wide_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? WIDE_OK : WIDE_ERR_CUDA; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool good_ptr(const void *p) { return p != nullptr && aligned16(p); }

bool good_group(int G) { return G == 64 || G == 128 || G == 256 || G == 512; }

// The M-axis (dynamic depth) case: one group spanning the whole grouped
// dimension (n_groups = 1, App. B "Implementation of GEMM-MN"), tile-aligned.
bool whole_width_group(int G, int width) { return G == width && G % 256 == 0; }

// Group sizes come from the tile-size set {2^k : k >= 4} (Sec. 3.1); members
// of the set outside {64..512} are valid but not implemented.
wide_status_t bad_group_status(int G) {
    return (G >= 16 && (G & (G - 1)) == 0) ? WIDE_ERR_UNSUPPORTED : WIDE_ERR_INVALID_ARG;
}

struct DeviceCtx {
    int num_sms;
    int *status;
};

wide_status_t device_ctx(DeviceCtx *ctx) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return WIDE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_num_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return WIDE_ERR_CUDA;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return WIDE_ERR_CUDA;
        g_status_ptr[dev] = static_cast<int *>(p);
        g_num_sms[dev] = n;
    }
    if (g_encode == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return WIDE_ERR_CUDA;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    ctx->num_sms = g_num_sms[dev];
    ctx->status = g_status_ptr[dev];
    return WIDE_OK;
}

// SM count that sizes the decode GEMM-K split (and so its workspace): the
// current device's, or 152 (GB300) when no device is visible.
int sizing_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
        return n;
    (void)cudaGetLastError();
    return 152;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous), box {64 cols, box_rows},
// 128-byte swizzle; out-of-range elements read as zero.
wide_status_t encode_bf16_2d(CUtensorMap *m, const void *base, long long rows, long long cols,
                             int box_rows) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? WIDE_OK : WIDE_ERR_CUDA;
}

// Decode (T <= 16) kernels, chosen by measurement on GB300 (8B FFN shapes):
// gate/up and q_proj stream weight rows on the CUDA cores up to 4 tokens and
// on the tensor cores above; down/o_proj run the GEMM-K kernel with the
// groups split over CTAs whenever N is a multiple of its 128-column tile.
constexpr int kDecodeMnCudaMaxT = 4;

bool decode_k_on_gemm_k(int N) { return N % 128 == 0; }

// Shared validation of GEMM-MN style calls; out features N grouped by G.
wide_status_t check_mn(const void *X, const void *W0, const void *W1, const void *mask,
                       const void *perm, const void *counts, int T, int K, int N, int G,
                       const void *out, bool need_w1) {
    if (!good_ptr(X) || !good_ptr(W0) || (need_w1 && !good_ptr(W1)) || !good_ptr(mask) ||
        !good_ptr(out))
        return WIDE_ERR_INVALID_ARG;
    if (T < 1 || K < 64 || N < 64 || K % 64 || N % 64) return WIDE_ERR_INVALID_ARG;
    if (!good_group(G) && !whole_width_group(G, N)) return bad_group_status(G);
    if (N % G) return WIDE_ERR_INVALID_ARG;
    if (N / G > wide::kMaxGroups) return WIDE_ERR_UNSUPPORTED;
    if (T > kDecodeMaxT && (!good_ptr(perm) || !good_ptr(counts))) return WIDE_ERR_INVALID_ARG;
    if ((perm != nullptr && !aligned16(perm)) || (counts != nullptr && !aligned16(counts)))
        return WIDE_ERR_INVALID_ARG;
    return WIDE_OK;
}

// Workspace a GEMM-K call cannot run without: fp32 partial sums of a split
// reduction (decode, and prefill grids smaller than the SMs).  The prefill
// tail split's workspace is optional (wide_gemm_k_workspace_size reports it).
size_t gemm_k_required_ws(int T, int K, int N, int G) {
    if (T < 1 || G <= 0 || K < G || K % G) return 0;
    if (T > kDecodeMaxT) return wide::gemm_k_split_workspace_bytes(T, K, N, G, sizing_sms());
    return decode_k_on_gemm_k(N) ? wide::gemm_k_decode_workspace_bytes(T, K, N, G, sizing_sms())
                                 : wide::decode_k_workspace_bytes(T, K, N, G);
}

wide_status_t check_k(const void *A, const void *W, const void *mask, int T, int K, int N, int G,
                      const void *out, const void *ws, size_t ws_bytes) {
    if (!good_ptr(A) || !good_ptr(W) || !good_ptr(mask) || !good_ptr(out))
        return WIDE_ERR_INVALID_ARG;
    if (T < 1 || K < 64 || N < 64 || K % 64 || N % 64) return WIDE_ERR_INVALID_ARG;
    if (!good_group(G) && !whole_width_group(G, K)) return bad_group_status(G);
    if (K % G) return WIDE_ERR_INVALID_ARG;
    if (K / G > wide::gemm_k_max_groups()) return WIDE_ERR_UNSUPPORTED;
    const size_t need = gemm_k_required_ws(T, K, N, G);
    if (need > 0 && (ws == nullptr || ws_bytes < need)) return WIDE_ERR_WORKSPACE;
    if (need > 0 && !aligned16(ws)) return WIDE_ERR_INVALID_ARG;
    return WIDE_OK;
}

wide_status_t run_mn(wide::MNMode mode, const uint16_t *X, const uint16_t *W0,
                     const uint16_t *W1, const uint8_t *mask, const int32_t *perm,
                     const int32_t *counts, int T, int K, int N, int G, uint16_t *out,
                     void *stream) {
    DeviceCtx ctx;
    wide_status_t st = device_ctx(&ctx);
    if (st != WIDE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool gate_up = mode == wide::MNMode::kGateUp;
    if (T <= kDecodeMnCudaMaxT && wide::decode_mn_smem_bytes(T, K, N / G) <= 200 * 1024) {
        wide::DecodeArgs a{X, W0, gate_up ? W1 : nullptr, mask, out, T, K, N, G};
        return from_cuda(wide::launch_decode_mn(mode, a, ctx.num_sms, s));
    }
    if (T <= kDecodeMaxT) {
        const int rt = wide::decode_tc_rows_per_item();
        CUtensorMap tmW0, tmW1, tmX;
        if ((st = encode_bf16_2d(&tmW0, W0, N, K, rt)) != WIDE_OK) return st;
        if ((st = encode_bf16_2d(&tmW1, gate_up ? W1 : W0, N, K, rt)) != WIDE_OK) return st;
        if ((st = encode_bf16_2d(&tmX, X, T, K, T < 16 ? T : 16)) != WIDE_OK) return st;
        wide::DecodeArgs a{X, W0, gate_up ? W1 : nullptr, mask, out, T, K, N, G};
        return from_cuda(
            wide::launch_decode_mn_tc(mode, tmW0, tmW1, tmX, a, ctx.status, ctx.num_sms, s));
    }
    if (perm == nullptr || counts == nullptr) return WIDE_ERR_INVALID_ARG;
    const int bn = gate_up ? (G == 64 ? 64 : 128) : (G == 64 ? 64 : G == 128 ? 128 : 256);
    CUtensorMap tmB0, tmB1;
    if ((st = encode_bf16_2d(&tmB0, W0, N, K, bn)) != WIDE_OK) return st;
    if ((st = encode_bf16_2d(&tmB1, gate_up ? W1 : W0, N, K, bn)) != WIDE_OK) return st;
    // Token bands of the tile order: keep one band of X (~32 MiB) resident in L2.
    const int ng = N / G;
    const long long x_bytes = static_cast<long long>(T) * K * 2;
    int bands = static_cast<int>((x_bytes + (32ll << 20) - 1) / (32ll << 20));
    bands = bands < 1 ? 1 : bands > 16 ? 16 : bands;
    while (bands > 1 && bands * ng > wide::kMaxGroups) --bands;
    wide::MNArgs a{X, perm, counts, out, T, K, N, G, bands, ctx.status};
    return from_cuda(wide::launch_gemm_mn(mode, bn, tmB0, tmB1, a, ctx.num_sms, s));
}

wide_status_t run_k(const uint16_t *A, const uint16_t *W, const uint8_t *mask, int T, int K,
                    int N, int G, uint16_t *out, void *ws, size_t ws_bytes, void *stream) {
    DeviceCtx ctx;
    wide_status_t st = device_ctx(&ctx);
    if (st != WIDE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T <= kDecodeMaxT && decode_k_on_gemm_k(N)) {
        CUtensorMap tmA, tmB;
        if ((st = encode_bf16_2d(&tmA, A, T, K, T < 16 ? T : 16)) != WIDE_OK) return st;
        if ((st = encode_bf16_2d(&tmB, W, N, K, wide::gemm_k_decode_bn(N))) != WIDE_OK) return st;
        wide::KArgs a{mask, out, T, K, N, G, ctx.status};
        a.a_rows = T < 16 ? T : 16;
        return from_cuda(
            wide::launch_gemm_k_decode(tmA, tmB, a, static_cast<float *>(ws), ctx.num_sms, s));
    }
    if (T <= kDecodeMaxT) {
        // a single group wider than the staged slice (whole-width G) does not fit
        if (wide::decode_k_smem_bytes(T, K, G) > 200 * 1024) return WIDE_ERR_UNSUPPORTED;
        wide::DecodeArgs a{A, W, nullptr, mask, out, T, K, N, G};
        return from_cuda(wide::launch_decode_k(a, static_cast<float *>(ws), s));
    }
    if (wide::gemm_k_prefill_splits(T, K, N, G, ctx.num_sms) > 1) {
        CUtensorMap tmA, tmB;
        if ((st = encode_bf16_2d(&tmA, A, T, K, 128)) != WIDE_OK) return st;
        if ((st = encode_bf16_2d(&tmB, W, N, K, wide::gemm_k_split_bn(N))) != WIDE_OK) return st;
        wide::KArgs a{mask, out, T, K, N, G, ctx.status};
        return from_cuda(
            wide::launch_gemm_k_split(tmA, tmB, a, static_cast<float *>(ws), ctx.num_sms, s));
    }
    const int bn = N % 256 == 0 ? 256 : N % 128 == 0 ? 128 : 64;
    CUtensorMap tmA, tmB;
    if ((st = encode_bf16_2d(&tmA, A, T, K, 128)) != WIDE_OK) return st;
    if ((st = encode_bf16_2d(&tmB, W, N, K, bn)) != WIDE_OK) return st;
    wide::KArgs a{mask, out, T, K, N, G, ctx.status};
    const size_t tail = wide::gemm_k_tail_workspace_bytes(T, K, N, G, ctx.num_sms);
    if (tail > 0 && ws != nullptr && ws_bytes >= tail && aligned16(ws))
        return from_cuda(wide::launch_gemm_k_tail(bn, tmA, tmB, a, static_cast<float *>(ws), ctx.num_sms, s));
    return from_cuda(wide::launch_gemm_k(bn, tmA, tmB, a, ctx.num_sms, s));
}

}  // namespace

// The cooperative reorder costs about 13 us whatever the size (the workspace
// memset and two grid barriers); one block per column grows with the column
// and leaves SMs idle when groups are few.  Measured on GB300 (us, coop vs
// column): 8 groups 13.8 vs 17.1 at T = 16384 and 14.1 vs 26.9 at T = 32768,
// but 13.5 vs 9.0 at T = 4096; 32 groups 20.2 vs 17.1 at T = 16384; 112
// groups 52.2 vs 27.3 at T = 32768, 62.4 vs 62.3 at T = 49152 and 75.0 vs
// 80.0 at T = 65536.
static bool reorder_prefers_coop(int T, int n_groups) {
    return T >= 65536 || (T >= 16384 && n_groups <= 16);
}

static bool reorder_coop_fits(int n_groups) { return wide::reorder_coop_smem_bytes(n_groups) <= 200 * 1024; }

extern "C" {

const char *wide_status_string(int status) {
    switch (status) {
        case WIDE_OK: return "WIDE_OK";
        case WIDE_ERR_INVALID_ARG: return "WIDE_ERR_INVALID_ARG";
        case WIDE_ERR_UNSUPPORTED: return "WIDE_ERR_UNSUPPORTED";
        case WIDE_ERR_WORKSPACE: return "WIDE_ERR_WORKSPACE";
        case WIDE_ERR_CUDA: return "WIDE_ERR_CUDA";
        case WIDE_ERR_TIMEOUT: return "WIDE_ERR_TIMEOUT";
        default: return "WIDE_ERR_UNKNOWN";
    }
}

int wide_version(void) { return kVersion; }

int wide_num_sms(void) {
    DeviceCtx ctx;
    return device_ctx(&ctx) == WIDE_OK ? ctx.num_sms : 0;
}



size_t wide_reorder_workspace_size(int T, int n_groups) {
    // the cooperative path's ballots and tile offsets, where it is the faster one
    if (T < 1 || n_groups < 1 || n_groups > 65535) return 0;
    if (!reorder_coop_fits(n_groups) || !reorder_prefers_coop(T, n_groups)) return 0;
    return wide::partition_workspace_bytes(T, n_groups);
}

wide_status_t wide_reorder_masks(const uint8_t *mask, int T, int n_groups, int32_t *perm,
                                 int32_t *counts, void *ws, size_t ws_bytes, void *stream) {
    if (!good_ptr(mask) || !good_ptr(perm) || !good_ptr(counts)) return WIDE_ERR_INVALID_ARG;
    if (T < 1 || n_groups < 1 || n_groups > 65535) return WIDE_ERR_INVALID_ARG;
    if (static_cast<long long>(T) * n_groups > (1ll << 40)) return WIDE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // a workspace large enough for the cooperative path selects it
    const size_t need = wide::partition_workspace_bytes(T, n_groups);
    if (ws != nullptr && ws_bytes >= need && aligned16(ws) && reorder_coop_fits(n_groups)) {
        DeviceCtx ctx;
        wide_status_t st = device_ctx(&ctx);
        if (st != WIDE_OK) return st;
        if (cudaMemsetAsync(ws, 0, 16, s) != cudaSuccess) return WIDE_ERR_CUDA;  // grid barrier counter
        const cudaError_t e = wide::launch_reorder_coop(mask, T, n_groups, perm, counts,
                                                        static_cast<uint32_t *>(ws), ctx.status,
                                                        ctx.num_sms, s);
        if (e != cudaErrorCooperativeLaunchTooLarge) return from_cuda(e);
        (void)cudaGetLastError();  // the grid cannot be resident: the one-kernel-per-column path
    }
    return from_cuda(wide::launch_reorder(mask, T, n_groups, perm, counts, s));
}

wide_status_t wide_router_masks(const uint16_t *X, const uint16_t *W1, const uint16_t *W2, int T,
                                int d_model, int r, int n_groups, uint8_t *mask, float *logits,
                                void *stream) {
    if (!good_ptr(X) || !good_ptr(W1) || !good_ptr(W2) || !good_ptr(mask)) return WIDE_ERR_INVALID_ARG;
    if (logits != nullptr && !aligned16(logits)) return WIDE_ERR_INVALID_ARG;
    if (T < 1 || d_model < 64 || d_model % 64 || r < 16 || r % 16 || n_groups < 1)
        return WIDE_ERR_INVALID_ARG;
    if (!wide::router_supported(r, n_groups)) return WIDE_ERR_UNSUPPORTED;
    DeviceCtx ctx;
    wide_status_t st = device_ctx(&ctx);
    if (st != WIDE_OK) return st;
    if (T <= kDecodeMaxT && d_model % 512 == 0) {
        // decode: a cluster of CUDA-core CTAs per token, each a slice of d_model
        // (a single 128-row tensor-core tile would walk d_model serially)
        wide::RouterArgs a{W2, mask, logits, T, d_model, r, n_groups, ctx.status};
        return from_cuda(wide::launch_router_decode(X, W1, a, static_cast<cudaStream_t>(stream)));
    }
    CUtensorMap tmX, tmW1;
    if ((st = encode_bf16_2d(&tmX, X, T, d_model, 128)) != WIDE_OK) return st;
    if ((st = encode_bf16_2d(&tmW1, W1, r, d_model, r)) != WIDE_OK) return st;
    wide::RouterArgs a{W2, mask, logits, T, d_model, r, n_groups, ctx.status};
    return from_cuda(wide::launch_router(tmX, tmW1, a, ctx.num_sms, static_cast<cudaStream_t>(stream)));
}

size_t wide_attn_decode_workspace_size(int B, int Hq, int d, int L_max) {
    if (B < 1 || Hq < 1 || d < 1 || L_max < 1) return 0;
    return wide::attn_decode_workspace_bytes(B, Hq, d, L_max);
}

wide_status_t wide_attn_decode(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                               const int32_t *lens, const uint8_t *mask, int B, int Hq, int Hk,
                               int d, int L_max, uint16_t *O, void *ws, size_t ws_bytes,
                               void *stream) {
    if (!good_ptr(Q) || !good_ptr(K) || !good_ptr(V) || !good_ptr(lens) || !good_ptr(mask) ||
        !good_ptr(O))
        return WIDE_ERR_INVALID_ARG;
    if (B < 1 || B > 65535 || Hq < 1 || Hk < 1 || Hk > 65535 || L_max < 1 || Hq % Hk)
        return WIDE_ERR_INVALID_ARG;
    if (!wide::attn_decode_supported(Hq, Hk, d, L_max)) return WIDE_ERR_UNSUPPORTED;
    const size_t need = wide::attn_decode_workspace_bytes(B, Hq, d, L_max);
    if (ws == nullptr || ws_bytes < need) return WIDE_ERR_WORKSPACE;
    if (!aligned16(ws)) return WIDE_ERR_INVALID_ARG;
    DeviceCtx ctx;
    wide_status_t st = device_ctx(&ctx);
    if (st != WIDE_OK) return st;
    float *ws_ml = static_cast<float *>(ws);
    float *ws_o = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) +
                                            wide::attn_decode_ml_bytes(B, Hq, L_max));
    const long long rows = static_cast<long long>(B) * Hk * L_max;
    if (rows > 0x7fffffffLL) return WIDE_ERR_UNSUPPORTED;  // TMA row coordinates are 32-bit
    CUtensorMap tmK, tmV;
    if ((st = encode_bf16_2d(&tmK, K, rows, d, 128)) != WIDE_OK) return st;
    if ((st = encode_bf16_2d(&tmV, V, rows, d, 128)) != WIDE_OK) return st;
    wide::AttnDecodeArgs a{Q,  K,  V,     lens, mask, O, ws_ml, ws_o, B, Hq, Hk, d, L_max,
                           wide::attn_decode_chunks(L_max), ctx.status};
    return from_cuda(wide::launch_attn_decode(tmK, tmV, a, static_cast<cudaStream_t>(stream)));
}

wide_status_t wide_attn_prefill(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                const int32_t *perm, const int32_t *counts, int B, int T, int Hq,
                                int Hk, int d, int causal, uint16_t *O, void *stream) {
    if (!good_ptr(Q) || !good_ptr(K) || !good_ptr(V) || !good_ptr(perm) || !good_ptr(counts) ||
        !good_ptr(O))
        return WIDE_ERR_INVALID_ARG;
    if (B < 1 || B > 65535 || T < 1 || Hq < 1 || Hq > 65535 || Hk < 1 || Hq % Hk)
        return WIDE_ERR_INVALID_ARG;
    if (!wide::attn_prefill_supported(Hq, Hk, d)) return WIDE_ERR_UNSUPPORTED;
    const long long rows = static_cast<long long>(B) * Hk * T;
    if (rows > 0x7fffffffLL - 128) return WIDE_ERR_UNSUPPORTED;  // TMA row coordinates are 32-bit
    DeviceCtx ctx;
    wide_status_t st = device_ctx(&ctx);
    if (st != WIDE_OK) return st;
    wide::AttnPrefillArgs a{Q, perm, counts, O, B, T, Hq, Hk, d, causal != 0, ctx.status};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // d = 128 runs on the tensor-core (tcgen05) kernel; both kernels take
    // 64-key tiles
    const bool tc = wide::attn_prefill_tc_supported(d);
    CUtensorMap tmK, tmV;
    if ((st = encode_bf16_2d(&tmK, K, rows, d, 64)) != WIDE_OK) return st;
    if ((st = encode_bf16_2d(&tmV, V, rows, d, 64)) != WIDE_OK) return st;
    return from_cuda(tc ? wide::launch_attn_prefill_tc(tmK, tmV, a, s)
                        : wide::launch_attn_prefill(tmK, tmV, a, s));
}

size_t wide_route_and_reorder_workspace_size(int T, int n_groups) {
    if (T <= kDecodeMaxT || n_groups < 1) return 0;
    return wide::route_reorder_workspace_bytes(T, n_groups);
}

wide_status_t wide_route_and_reorder(const uint16_t *X, const uint16_t *W1, const uint16_t *W2,
                                     int T, int d_model, int r, int n_groups, uint8_t *mask,
                                     int32_t *perm, int32_t *counts, void *ws, size_t ws_bytes,
                                     void *stream) {
    if (!good_ptr(perm) || !good_ptr(counts) || n_groups > 65535) return WIDE_ERR_INVALID_ARG;
    const size_t fused_ws = wide_route_and_reorder_workspace_size(T, n_groups);
    if (fused_ws > 0 && ws != nullptr && ws_bytes >= fused_ws) {
        // one cooperative launch: router, then the reorder of its mask
        if (!good_ptr(X) || !good_ptr(W1) || !good_ptr(W2) || !good_ptr(mask) || !aligned16(ws))
            return WIDE_ERR_INVALID_ARG;
        if (d_model < 64 || d_model % 64 || r < 16 || r % 16) return WIDE_ERR_INVALID_ARG;
        if (!wide::router_supported(r, n_groups)) return WIDE_ERR_UNSUPPORTED;
        DeviceCtx ctx;
        wide_status_t st = device_ctx(&ctx);
        if (st != WIDE_OK) return st;
        CUtensorMap tmX, tmW1;
        if ((st = encode_bf16_2d(&tmX, X, T, d_model, 128)) != WIDE_OK) return st;
        if ((st = encode_bf16_2d(&tmW1, W1, r, d_model, r)) != WIDE_OK) return st;
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        if (cudaMemsetAsync(ws, 0, 16, s) != cudaSuccess) return WIDE_ERR_CUDA;  // grid barrier counter
        wide::RouterArgs a{W2, mask, nullptr, T, d_model, r, n_groups, ctx.status};
        a.perm = perm;
        a.counts = counts;
        a.ws = static_cast<uint32_t *>(ws);
        const cudaError_t e = wide::launch_route_reorder(tmX, tmW1, a, ctx.num_sms, s);
        if (e != cudaErrorCooperativeLaunchTooLarge) return from_cuda(e);
        // the grid could not be co-resident (e.g. a partitioned GPU): two launches
        (void)cudaGetLastError();
    }
    wide_status_t st = wide_router_masks(X, W1, W2, T, d_model, r, n_groups, mask, nullptr, stream);
    if (st != WIDE_OK) return st;
    return wide_reorder_masks(mask, T, n_groups, perm, counts, ws, ws_bytes, stream);
}

wide_status_t wide_gemm_mn_gate_up(const uint16_t *X, const uint16_t *W_gate,
                                   const uint16_t *W_up, const uint8_t *mask,
                                   const int32_t *perm, const int32_t *counts, int T, int d_model,
                                   int d_ffn, int G, uint16_t *H, void *stream) {
    wide_status_t st = check_mn(X, W_gate, W_up, mask, perm, counts, T, d_model, d_ffn, G, H, true);
    if (st != WIDE_OK) return st;
    return run_mn(wide::MNMode::kGateUp, X, W_gate, W_up, mask, perm, counts, T, d_model, d_ffn,
                  G, H, stream);
}

wide_status_t wide_proj_mn(const uint16_t *X, const uint16_t *W, const uint8_t *mask,
                           const int32_t *perm, const int32_t *counts, int T, int K, int N, int G,
                           uint16_t *Y, void *stream) {
    wide_status_t st = check_mn(X, W, nullptr, mask, perm, counts, T, K, N, G, Y, false);
    if (st != WIDE_OK) return st;
    return run_mn(wide::MNMode::kPlain, X, W, nullptr, mask, perm, counts, T, K, N, G, Y, stream);
}

size_t wide_gemm_k_workspace_size(int T, int K, int N, int G) {
    // Decode, and prefill too small to fill the SMs, sum fp32 partials of the
    // split reduction dimension (required).  Large prefill reduces in TMEM; when
    // its last wave of output tiles would leave half of the SMs idle, an
    // optional workspace lets that wave's tiles be split (the tail split).
    const size_t need = gemm_k_required_ws(T, K, N, G);
    if (need > 0 || T <= kDecodeMaxT || T < 1 || G <= 0 || K < G || K % G) return need;
    return wide::gemm_k_tail_workspace_bytes(T, K, N, G, sizing_sms());
}

wide_status_t wide_gemm_k_down(const uint16_t *H, const uint16_t *W_down, const uint8_t *mask,
                               const int32_t *perm, const int32_t *counts, int T, int d_ffn,
                               int d_model, int G, uint16_t *Y, void *ws, size_t ws_bytes,
                               void *stream) {
    (void)perm;
    (void)counts;
    wide_status_t st = check_k(H, W_down, mask, T, d_ffn, d_model, G, Y, ws, ws_bytes);
    if (st != WIDE_OK) return st;
    return run_k(H, W_down, mask, T, d_ffn, d_model, G, Y, ws, ws_bytes, stream);
}

wide_status_t wide_proj_k(const uint16_t *A, const uint16_t *W, const uint8_t *mask,
                          const int32_t *perm, const int32_t *counts, int T, int K, int N, int G,
                          uint16_t *Y, void *ws, size_t ws_bytes, void *stream) {
    (void)perm;
    (void)counts;
    wide_status_t st = check_k(A, W, mask, T, K, N, G, Y, ws, ws_bytes);
    if (st != WIDE_OK) return st;
    return run_k(A, W, mask, T, K, N, G, Y, ws, ws_bytes, stream);
}

wide_status_t wide_device_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return WIDE_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof v) != cudaSuccess) return WIDE_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero) != cudaSuccess)
            return WIDE_ERR_CUDA;
    }
    return static_cast<wide_status_t>(v);
}

}  // extern "C"
