/*
 * wide.h -- C ABI of libwide.so: GB300 (sm_103a) kernels for the hot path of
 * WIDE token-level dynamic width pruning ("WIDE: Boosting Adaptive LLM
 * Inference via Token-level Dynamic Width Pruning", arXiv 2607.28418).
 *
 * Notation (Sec. 3.3): a projection is C = A B^T with A in R^{M x K} (token
 * rows; batch and sequence flattened into M, called T here), B in R^{N x K}
 * (nn.Linear weight layout, [out_features, in_features], K contiguous).
 * A routing mask M in {0,1}^{T x n_groups} (row-major uint8, any nonzero byte
 * means active) selects, per token, contiguous groups of G channels:
 *   - GEMM-MN: groups tile the OUTPUT features N (q_proj, gate/up), Eq. 2-3;
 *   - GEMM-K : groups tile the REDUCTION dimension K (o_proj, down), Eq. 21.
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  bf16
 *     tensors are passed as their raw 16-bit patterns (uint16_t), row-major
 *     and densely packed.  Every pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *     enqueue work on it: no host synchronisation, no device-to-host copy, no
 *     allocation.  Nothing is returned to the host through memory.
 *   - Shapes: T >= 1; G in {64, 128, 256, 512}; every feature dimension is a
 *     multiple of 64 and of G where it is grouped.  G may also equal the whole
 *     grouped dimension (N for GEMM-MN, K for GEMM-K) when that is a multiple
 *     of 256: one group per token, the M-axis (dynamic depth) special case
 *     N_G = 1 of App. B ("Implementation of GEMM-MN"); the mask is [T, 1].
 *   - Outputs are fully overwritten (never accumulated into): MN outputs hold
 *     exact zeros in inactive (token, group) blocks; K outputs of a token with
 *     no active group are zero.  K calls ignore the values of A inside
 *     inactive groups (Eq. 21 multiplies them by M).
 *   - Errors: argument errors are detected on the host before anything is
 *     launched (WIDE_ERR_INVALID_ARG / WIDE_ERR_UNSUPPORTED).  A failed
 *     launch returns WIDE_ERR_CUDA.  Kernels never trap: a pipeline wait that
 *     exceeds its time limit records WIDE_ERR_TIMEOUT in a device status word
 *     that wide_device_status() reads back, and a kernel that finds itself
 *     launched without the thread-block cluster it needs (as a tool that
 *     re-launches graph nodes one by one may do) records WIDE_ERR_CUDA there
 *     and writes no output.
 */
#ifndef WIDE_H
#define WIDE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    WIDE_OK = 0,
    WIDE_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad shape          */
    WIDE_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. G = 32)     */
    WIDE_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required  */
    WIDE_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed           */
    WIDE_ERR_TIMEOUT = 5       /* a device-side wait gave up (see above)      */
} wide_status_t;

/* Human-readable name of a status code (static string, never NULL). */
const char *wide_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
int wide_version(void);

/* Number of SMs the persistent kernels size their grids to (device of the
 * calling thread); 0 if no device is visible. */
int wide_num_sms(void);

/*
 * Mask reordering -- Sec. 3.3 Eq. 7 and App. B Algorithm 1: every routing
 * column M[:, g] is SortDesc-ed independently, packing the active rows into
 * a prefix.  The sort is stable: perm[g][0 .. counts[g]) lists the active
 * rows of group g in ascending order, perm[g][counts[g] .. T) the inactive
 * rows in ascending order, so M[perm[g][j], g] != 0 exactly when
 * j < counts[g] (the index identity of App. B).
 *   mask   : uint8 [T, n_groups] row-major (device)
 *   perm   : int32 [n_groups, T] group-major (device, written)
 *   counts : int32 [n_groups]    (device, written)
 *   ws     : optional.  With 16 + 20 * ceil(T/128) * n_groups bytes (16-byte
 *            aligned), the partition runs as one cooperative kernel launch
 *            (after an 8-byte memset of the workspace) that reads the mask
 *            rows coalesced and ballots each group over 32-token warps;
 *            otherwise (ws NULL or smaller, or a grid that cannot be
 *            resident) one block per column walks its column.  Same result
 *            either way.  wide_reorder_workspace_size() returns that size
 *            where the cooperative launch measured faster (T >= 65536, or
 *            T >= 16384 with n_groups <= 16), else 0.
 * Bit-exact and deterministic.  T <= 2^31 - 1, 1 <= n_groups <= 65535.
 */
wide_status_t wide_reorder_masks(const uint8_t *mask, int T, int n_groups,
                                 int32_t *perm, int32_t *counts,
                                 void *ws, size_t ws_bytes, void *stream);
size_t wide_reorder_workspace_size(int T, int n_groups);

/*
 * Router, inference branch -- Sec. 3.1 "Routing Components", Eq. 4-5:
 *   z[t, j]    = sum_d X[t,d] W1[j,d]              (bottleneck, j < r)
 *   R[t, g, c] = sum_j z[t,j] W2[2g+c, j]          (X W1 W2 reshaped to [T, N_G, 2])
 *   mask[t, g] = 1 when argmax_c R[t,g,c] = 0 (class 0 executes), i.e.
 *                R[t,g,0] >= R[t,g,1]; a tie executes (first maximum).
 *   X      : bf16 [T, d_model]
 *   W1     : bf16 [r, d_model]      (the page's D x r matrix, stored [out, in])
 *   W2     : bf16 [2 n_groups, r]   (the page's r x 2N_G matrix, stored [out, in])
 *   mask   : uint8 [T, n_groups], written (0 or 1)
 *   logits : float [T, 2 n_groups] (column 2g + c), written when not NULL
 * z is accumulated in fp32 (by the tensor cores, or for T <= 16 and
 * d_model % 512 == 0 by a cluster of 8 CUDA-core blocks per token, one slice
 * of d_model each) and the logits are fp32 FMA sums in ascending j; the
 * decision is taken on those fp32 logits.
 * r in {16, 32, 64}; d_model % 64 == 0; 2 * n_groups * r * 2 <= 65536 bytes
 * (else WIDE_ERR_UNSUPPORTED).
 */
wide_status_t wide_router_masks(const uint16_t *X, const uint16_t *W1, const uint16_t *W2,
                                int T, int d_model, int r, int n_groups, uint8_t *mask,
                                float *logits, void *stream);

/*
 * Routed decode attention -- App. B "Implementation of Attention" (decoding:
 * routing is checked per block, split online softmax) with the GQA-aligned
 * groups of Sec. 3.1 Eq. 2 (G = (Hq/Hk) d, so group g is KV head g and its
 * Hq/Hk query heads).  One query token per sequence b:
 *   O[b,h,:] = mask[b,g] * sum_j softmax_j(Q[b,h,:] . K[b,g,j,:] / sqrt(d)) V[b,g,j,:]
 * over the first lens[b] cached keys (g = h / (Hq/Hk)); an inactive group or
 * lens[b] <= 0 gives zeros, and the cache of an inactive group is not read.
 *   Q    : bf16 [B, Hq, d]           K, V : bf16 [B, Hk, L_max, d]
 *   lens : int32 [B] (device; values are clamped to [0, L_max])
 *   mask : uint8 [B, Hk]             O    : bf16 [B, Hq, d] (written)
 *   ws   : wide_attn_decode_workspace_size(B, Hq, d, L_max) bytes of device
 *          memory (fp32 per-chunk partial sums), 16-byte aligned
 * d in {64, 128}; Hq/Hk in {1, 2, 4, 8}; L_max <= 130816 (1022 chunks of 128
 * keys) (else WIDE_ERR_UNSUPPORTED); B, Hk <= 65535.
 */
wide_status_t wide_attn_decode(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                               const int32_t *lens, const uint8_t *mask, int B, int Hq, int Hk,
                               int d, int L_max, uint16_t *O, void *ws, size_t ws_bytes,
                               void *stream);
size_t wide_attn_decode_workspace_size(int B, int Hq, int d, int L_max);

/*
 * Routed prefill attention -- App. B "Implementation of Attention", prefill
 * (Algorithm 4), with the GQA-aligned groups of Sec. 3.1 Eq. 2: query head h
 * reads KV head g = h / (Hq/Hk), which is also its routing group.
 *   O[b,t,h,:] = mask[b,t,g] * sum_j softmax_j(Q[b,t,h,:] . K[b,g,j,:] / sqrt(d)) V[b,g,j,:]
 * over keys j <= t (causal != 0) or all T keys; inactive rows are zero.
 *   Q      : bf16 [B, T, Hq, d]          K, V : bf16 [B, Hk, T, d]
 *   perm, counts : for every sequence b, wide_reorder_masks() of its mask
 *            mask[b] ([T, Hk]): perm [B, Hk, T] int32, counts [B, Hk] int32
 *   O      : bf16 [B, T, Hq, d] (every element written)
 * Scores and P V run on the tensor cores (tcgen05 with S and O in TMEM for
 * d = 128, the warp-level instruction for d = 64; bf16 in, fp32 accumulate,
 * P rounded to bf16); the softmax is online in fp32.
 * d in {64, 128} (else WIDE_ERR_UNSUPPORTED); B, Hq <= 65535.
 */
wide_status_t wide_attn_prefill(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                const int32_t *perm, const int32_t *counts, int B, int T, int Hq,
                                int Hk, int d, int causal, uint16_t *O, void *stream);

/*
 * The router followed by the mask reordering of that mask (Eq. 4-5 then
 * Eq. 7), both enqueued on `stream`: mask, perm and counts are ready for the
 * GEMM calls.  Arguments as for wide_router_masks and wide_reorder_masks.
 *   ws : with at least wide_route_and_reorder_workspace_size(T, n_groups)
 *        bytes (16-byte aligned; nonzero only for T > 16), the two run as
 *        one cooperative kernel launch (after an 8-byte memset of the
 *        workspace): each CTA routes its 128-token tiles, and after grid
 *        barriers the CTAs scan the per-tile active counts and place their
 *        own tokens.  With a smaller or NULL workspace, or T <= 16, or when
 *        the device cannot keep the whole grid resident, the router and the
 *        reorder kernel run one after the other.  Same results either way
 *        (perm and counts bit-identical).
 */
size_t wide_route_and_reorder_workspace_size(int T, int n_groups);
wide_status_t wide_route_and_reorder(const uint16_t *X, const uint16_t *W1, const uint16_t *W2,
                                     int T, int d_model, int r, int n_groups, uint8_t *mask,
                                     int32_t *perm, int32_t *counts, void *ws, size_t ws_bytes,
                                     void *stream);

/*
 * FFN gate/up projection with fused activation -- Sec. 3.1 Eq. 3 (GEMM-MN,
 * App. B Algorithm 2):
 *   H[t, f] = M[t, f/G] * silu(X[t,:] . W_gate[f,:]) * (X[t,:] . W_up[f,:])
 * with silu(a) = a * sigmoid(a), fp32 accumulation, bf16 (RNE) output.
 *   X        : bf16 [T, d_model]
 *   W_gate   : bf16 [d_ffn, d_model];  W_up : bf16 [d_ffn, d_model]
 *   mask     : uint8 [T, d_ffn/G]
 *   perm, counts : output of wide_reorder_masks() for this mask; may be NULL
 *              when T <= 16 (the decode path reads the mask directly)
 *   H        : bf16 [T, d_ffn] (written; inactive blocks are 0)
 * d_model % 64 == 0, d_ffn % G == 0.
 */
wide_status_t wide_gemm_mn_gate_up(const uint16_t *X, const uint16_t *W_gate,
                                   const uint16_t *W_up, const uint8_t *mask,
                                   const int32_t *perm, const int32_t *counts,
                                   int T, int d_model, int d_ffn, int G,
                                   uint16_t *H, void *stream);

/*
 * FFN down projection -- Sec. 3.1 Eq. 3 / App. B Eq. 21 (GEMM-K):
 *   Y[t, n] = sum_g M[t,g] sum_{f in [gG, (g+1)G)} H[t,f] * W_down[n,f]
 *   H      : bf16 [T, d_ffn]   (values inside inactive groups are ignored)
 *   W_down : bf16 [d_model, d_ffn]
 *   mask   : uint8 [T, d_ffn/G]; perm/counts as above (may be NULL)
 *   Y      : bf16 [T, d_model] (written)
 *   ws     : device workspace (16-byte aligned) of
 *            wide_gemm_k_workspace_size(T, d_ffn, d_model, G) bytes.  For
 *            decode and for batches too short to fill the GPU it is
 *            required (WIDE_ERR_WORKSPACE without it).  For larger batches it
 *            is optional: with it, the output tiles of a last wave that would
 *            leave at least half of the SMs idle are cut into 2-4 equal
 *            shares of their live groups (fp32 partials, added in order by
 *            a second kernel); with ws NULL or smaller, every tile is
 *            reduced whole.  NULL is accepted when the size is 0.
 * fp32 accumulation in ascending group order (when the groups are split over
 * CTAs -- decode, short batches, the tail tiles above -- ascending within
 * each share, then the shares in order); deterministic for a given device.
 */
wide_status_t wide_gemm_k_down(const uint16_t *H, const uint16_t *W_down,
                               const uint8_t *mask, const int32_t *perm,
                               const int32_t *counts, int T, int d_ffn,
                               int d_model, int G, uint16_t *Y, void *ws,
                               size_t ws_bytes, void *stream);

/*
 * Plain GEMM-MN (q_proj over GQA head groups, Sec. 3.1 Eq. 2; the M-axis
 * case is n_groups = N/G = 1, Sec. 3.3):
 *   Y[t, n] = M[t, n/G] * sum_k X[t,k] W[n,k]
 *   X : bf16 [T, K];  W : bf16 [N, K];  mask : uint8 [T, N/G];  Y : bf16 [T, N]
 */
wide_status_t wide_proj_mn(const uint16_t *X, const uint16_t *W,
                           const uint8_t *mask, const int32_t *perm,
                           const int32_t *counts, int T, int K, int N, int G,
                           uint16_t *Y, void *stream);

/*
 * Plain GEMM-K (o_proj over GQA head groups, Sec. 3.1 Eq. 2; App. B Eq. 21):
 *   Y[t, n] = sum_g M[t,g] sum_{k in [gG, (g+1)G)} A[t,k] W[n,k]
 *   A : bf16 [T, K];  W : bf16 [N, K];  mask : uint8 [T, K/G];  Y : bf16 [T, N]
 *   ws as for wide_gemm_k_down.
 */
wide_status_t wide_proj_k(const uint16_t *A, const uint16_t *W,
                          const uint8_t *mask, const int32_t *perm,
                          const int32_t *counts, int T, int K, int N, int G,
                          uint16_t *Y, void *ws, size_t ws_bytes, void *stream);

/* Workspace bytes a GEMM-K call takes for these sizes on the current device
 * (0 = none): fp32 partial sums when the groups are split over CTAs -- T <= 16,
 * a batch whose output-tile grid would leave SMs idle (both required), or the
 * tiles of a mostly idle last wave of a larger batch (optional, see
 * wide_gemm_k_down). */
size_t wide_gemm_k_workspace_size(int T, int K, int N, int G);

/*
 * Allocation-free decode GEMM-K (T <= 16).  No counterpart in the paper: an
 * addition of this library for callers that cannot allocate device memory
 * (a memory planner that owns every device allocation, a plugin host that
 * provides no workspace, or a path where a cudaMalloc would synchronise).
 *
 * Computes what wide_gemm_k_down / wide_proj_k compute for T <= 16:
 *   Y[t, n] = sum_g M[t,g] sum_{k in [gG,(g+1)G)} A[t,k] W[n,k]
 * (A: bf16 [T, K]; W: bf16 [N, K]; mask: uint8 [T, K/G]; Y: bf16 [T, N]),
 * to the same tolerance, on the CUDA-core split-K decode kernel (its
 * summation order, and so the last bits, can differ from the workspace
 * entry points', which use the tensor-core kernel when N % 128 == 0).  Its
 * fp32 partial sums live in a fixed array of WIDE_NOALLOC_SCRATCH_BYTES
 * inside the library (held by every GPU that loads the library until the
 * process exits) instead of a caller workspace.  Nothing is allocated or freed by this call.
 *   - Sizes whose partial sums (splits x T x N x 4 bytes; 1.3 MB for
 *     T = 16, K = 14336, N = 4096, G = 128) exceed the array return
 *     WIDE_ERR_WORKSPACE; T > 16 returns WIDE_ERR_INVALID_ARG.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) and caches it; make that first call before any
 *     stream capture on that device.
 *   - Every call shares the one array; the partial sums of a call are fully
 *     written before they are read, so nothing needs clearing between
 *     calls.  Calls whose kernels overlap on the GPU (e.g. issued on two
 *     streams without ordering) race on the array: order them on one stream.
 */
#define WIDE_NOALLOC_SCRATCH_BYTES (4u << 20)
wide_status_t wide_gemm_k_decode_noalloc(const uint16_t *A, const uint16_t *W,
                                         const uint8_t *mask, int T, int K, int N, int G,
                                         uint16_t *Y, void *stream);

/*
 * Device status word: synchronises `stream`, returns WIDE_OK or the first
 * device-side failure recorded since the last call (WIDE_ERR_TIMEOUT), and
 * clears it.  This is the only call that synchronises.
 */
wide_status_t wide_device_status(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* WIDE_H */
