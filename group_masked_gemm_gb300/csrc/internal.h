// internal.h -- host-side launchers shared between the C-ABI layer (api.cu)
// and the kernel translation units.  Arguments are validated by api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace wide {

// GEMM-MN flavours: plain projection or fused silu(gate) * up.
enum class MNMode { kPlain = 0, kGateUp = 1 };

struct MNArgs {
    const uint16_t *a_rows; // bf16 [T, K] token-row operand, gathered through perm
    const int32_t *perm;    // [n_groups, T]
    const int32_t *counts;  // [n_groups]
    uint16_t *out;          // bf16 [T, n_out]
    int T, K, n_out, G;
    int bands;              // token bands of the tile order (bands * n_groups <= kMaxGroups)
    int *status;
};

struct KArgs {
    const uint8_t *mask;  // [T, n_groups]
    uint16_t *out;        // bf16 [T, N] (when partial == nullptr)
    int T, K, N, G;
    int *status;
    // Decode only: item (n-tile, split s) reduces the s-th equal share of the
    // live groups and writes fp32 partial[s][T][N].
    float *partial = nullptr;
    int splits = 1;
    int a_rows = 128;  // rows of the token-row TMA box (<= 128)
    // Prefill tail split (n_direct >= 0): the first n_direct items write Y
    // directly; each later item is cut into tail_splits equal shares of its
    // live groups, share s of the j-th such item writing fp32 partial sums
    // to tail_partial[j * tail_splits + s][BM][BN].
    int n_direct = -1;
    int tail_splits = 1;
    float *tail_partial = nullptr;
};

struct RouterArgs {
    const uint16_t *W2;  // bf16 [2 n_groups, r]
    uint8_t *mask;       // [T, n_groups]
    float *logits;       // [T, 2 n_groups] or nullptr
    int T, D, r, n_groups;
    int *status;
    int stages = 0;  // pipeline depth, set by the launcher
    // fused reorder (route_and_reorder in one launch); null for the router alone
    int32_t *perm = nullptr;     // [n_groups, T]
    int32_t *counts = nullptr;   // [n_groups]
    uint32_t *ws = nullptr;      // route_reorder_workspace_bytes(T, n_groups), barrier word zeroed
};

struct AttnDecodeArgs {
    const uint16_t *Q;      // bf16 [B, Hq, d]
    const uint16_t *K, *V;  // bf16 [B, Hk, L_max, d]
    const int32_t *lens;    // [B] cached keys per sequence
    const uint8_t *mask;    // [B, Hk] one routing group per KV head
    uint16_t *O;            // bf16 [B, Hq, d]
    float *ws_ml;           // [B, Hq, n_chunks][2]: chunk max and sum
    float *ws_o;            // [B, Hq, n_chunks][d]: chunk numerators
    int B, Hq, Hk, d, L_max, n_chunks;
    int *status;
};

struct AttnPrefillArgs {
    const uint16_t *Q;       // bf16 [B, T, Hq, d]
    const int32_t *perm;     // [B, Hk, T]: per sequence, the stable partition of mask[b] [T, Hk]
    const int32_t *counts;   // [B, Hk]
    uint16_t *O;             // bf16 [B, T, Hq, d]
    int B, T, Hq, Hk, d, causal;
    int *status;
};

struct DecodeArgs {
    const uint16_t *x;     // bf16 [T, K]
    const uint16_t *w0;    // bf16 [N, K]  (gate, or the only weight)
    const uint16_t *w1;    // bf16 [N, K]  (up) or nullptr
    const uint8_t *mask;   // [T, n_groups]
    uint16_t *out;         // bf16 [T, N]
    int T, K, N, G;
};

// Largest n_groups the GEMM kernels keep in shared memory.
constexpr int kMaxGroups = 1024;

cudaError_t launch_reorder(const uint8_t *mask, int T, int n_groups, int32_t *perm,
                           int32_t *counts, cudaStream_t s);
// Cooperative reorder with coalesced mask reads: ws holds
// partition_workspace_bytes(T, n_groups) bytes, its first 16 zeroed.
size_t reorder_coop_smem_bytes(int n_groups);
cudaError_t launch_reorder_coop(const uint8_t *mask, int T, int n_groups, int32_t *perm, int32_t *counts,
                                uint32_t *ws, int *status, int num_sms, cudaStream_t s);

// tmB0/tmB1: tiled maps over the weights [n_out, K] (box 64 x bn, 128-B swizzle)
cudaError_t launch_gemm_mn(MNMode mode, int bn, const CUtensorMap &tmB0, const CUtensorMap &tmB1,
                           const MNArgs &a, int num_sms, cudaStream_t s);

// tmA: tiled map over the token-row operand [T, K] (box 64 x 128)
// tmB: tiled map over the weights [N, K] (box 64 x bn)
// Prefill tail split: workspace bytes (0 = the split does not apply) and the
// launch (the GEMM-K kernel, then a finalize that adds the shares in order).
size_t gemm_k_tail_workspace_bytes(int T, int K, int N, int G, int num_sms);
cudaError_t launch_gemm_k_tail(int bn, const CUtensorMap &tmA, const CUtensorMap &tmB, const KArgs &a,
                               float *ws, int num_sms, cudaStream_t s);
cudaError_t launch_gemm_k(int bn, const CUtensorMap &tmA, const CUtensorMap &tmB,
                          const KArgs &a, int num_sms, cudaStream_t s);

// Decode (T <= 16) GEMM-K on the GEMM-K kernel with the groups split over
// CTAs: tmA box 64 x min(T,16) (a.a_rows), tmB box 64 x 128, N % 128 == 0;
// ws: gemm_k_decode_workspace_bytes(T, K, N, G, num_sms) of fp32 partials.
int gemm_k_decode_bn(int N);
int gemm_k_decode_splits(int T, int K, int N, int G, int num_sms);
// Prefill (T > 16) whose output-tile grid is too small for the SMs: the
// groups are split over CTAs (same share rule and fp32 partials as decode)
// when gemm_k_prefill_splits() > 1; tmB box 64 x gemm_k_split_bn(N) rows;
// ws: gemm_k_split_workspace_bytes.
int gemm_k_split_bn(int N);
int gemm_k_prefill_splits(int T, int K, int N, int G, int num_sms);
size_t gemm_k_split_workspace_bytes(int T, int K, int N, int G, int num_sms);
cudaError_t launch_gemm_k_split(const CUtensorMap &tmA, const CUtensorMap &tmB, const KArgs &a,
                                float *ws, int num_sms, cudaStream_t s);
size_t gemm_k_decode_workspace_bytes(int T, int K, int N, int G, int num_sms);
cudaError_t launch_gemm_k_decode(const CUtensorMap &tmA, const CUtensorMap &tmB, const KArgs &a,
                                 float *ws, int num_sms, cudaStream_t s);

cudaError_t launch_decode_mn(MNMode mode, const DecodeArgs &a, int num_sms, cudaStream_t s);
// ws: fp32 partial sums, decode_k_workspace_bytes(T, K, N, G) bytes; the
// kernel stages decode_k_smem_bytes(T, K, G) of shared memory.
size_t decode_k_smem_bytes(int T, int K, int G);

// Routed decode attention: d in {64, 128}, Hq/Hk in {1, 2, 4, 8}, at most
// 1022 chunks of 128 keys.
bool attn_decode_supported(int Hq, int Hk, int d, int L_max);
int attn_decode_chunks(int L_max);
size_t attn_decode_ml_bytes(int B, int Hq, int L_max);
size_t attn_decode_workspace_bytes(int B, int Hq, int d, int L_max);
// tmK, tmV: [B * Hk * L_max, d] views of the caches, box 64 x 128, 128-byte swizzle.
cudaError_t launch_attn_decode(const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnDecodeArgs &a,
                               cudaStream_t s);

// Routed prefill attention: tmK, tmV are [B * Hk * T, d] views of K and V,
// box 64 x 64, 128-byte swizzle; d in {64, 128}.
bool attn_prefill_supported(int Hq, int Hk, int d);
cudaError_t launch_attn_prefill(const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnPrefillArgs &a,
                                cudaStream_t s);

// Routed prefill attention on tcgen05 (d = 128): tmK, tmV are [B * Hk * T, d]
// views of K and V with box 64 x 64, 128-byte swizzle.
bool attn_prefill_tc_supported(int d);
cudaError_t launch_attn_prefill_tc(const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnPrefillArgs &a,
                                   cudaStream_t s);

// Router (Eq. 4-5): tmX box 64 x 128 token rows of X [T, D]; tmW1 box 64 x r
// rows of W1 [r, D].  r in {16, 32, 64}; W2 (2 n_groups x r bf16) <= 64 KB.
bool router_supported(int r, int n_groups);
// Decode router (T <= 16) on CUDA cores: a cluster of 8 CTAs per token, each
// a slice of d; needs D % 512 == 0 and r <= 64.
cudaError_t launch_router_decode(const uint16_t *X, const uint16_t *W1, const RouterArgs &a,
                                 cudaStream_t s);
// Router and mask reordering in one cooperative launch (T > 16): a.perm,
// a.counts and a.ws set; the first 16 bytes of a.ws must be zero (a grid
// barrier counter).
size_t route_reorder_workspace_bytes(int T, int n_groups);
cudaError_t launch_route_reorder(const CUtensorMap &tmX, const CUtensorMap &tmW1, const RouterArgs &a,
                                 int num_sms, cudaStream_t s);
cudaError_t launch_router(const CUtensorMap &tmX, const CUtensorMap &tmW1, const RouterArgs &a,
                          int num_sms, cudaStream_t s);
cudaError_t launch_decode_k(const DecodeArgs &a, float *ws, cudaStream_t s);
size_t decode_k_workspace_bytes(int T, int K, int N, int G);
size_t decode_mn_smem_bytes(int T, int K, int n_groups);
cudaError_t launch_decode_k_finalize(const float *ws, int splits, int TN, uint16_t *out,
                                     cudaStream_t s);

// Tensor-core decode (T <= 16): weight rows on the MMA's M side, tokens on N.
// tmW0/tmW1: weight maps, box 64 x decode_tc_rows_per_item(); tmX: token rows
// [T, K], box 64 x min(T, 16).  GEMM-K: tmW box 64 x 128 (N % 128 == 0),
// tmA: the token rows [T, K], box 64 x min(T, 16).
int decode_tc_rows_per_item();
cudaError_t launch_decode_mn_tc(MNMode mode, const CUtensorMap &tmW0, const CUtensorMap &tmW1,
                                const CUtensorMap &tmX, const DecodeArgs &a, int *status,
                                int num_sms, cudaStream_t s);

}  // namespace wide
