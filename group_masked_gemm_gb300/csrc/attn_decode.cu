// attn_decode.cu -- routed decode attention (WIDE, App. B "Implementation of
// Attention", decoding paragraph; Sec. 3.1 Eq. 2).
//
// The attention groups are GQA-aligned (G = (Hq/Hk) d), so routing group g
// of a sequence is KV head g with its Hq/Hk query heads.  For one query token
// per sequence b:
//   O[b,h,:] = M[b,g] * softmax_j(q[b,h,:] . K[b,g,j,:] / sqrt(d)) V[b,g,j,:]
// over the lens[b] cached keys.  Decode attention is bound by HBM reads of the
// KV cache, and an inactive (sequence, group) pair never reads its cache.
//
// Split online softmax in two kernels:
//   attn_partial: one CTA per (128-key chunk, KV head, sequence); a chunk of
//     an inactive group, or past lens[b], returns without a read.  K and V of
//     the chunk arrive by TMA (128-byte swizzle) into shared memory.  The two
//     products are 16 x 128 x 128 per chunk (the group's <= 8 query heads on
//     the M side), far below tcgen05's smallest tile, so they run on the
//     warp-level tensor-core instruction (mma.sync m16n8k16, bf16 in, fp32
//     accumulate) with ldmatrix reads of the swizzled tiles: S = Q K^T, the
//     chunk softmax in fp32, then O = P V with P rounded to bf16.  Each
//     head's chunk maximum m, sum l = sum exp(s - m) and o = sum exp(s - m) v
//     go to the workspace.
//   attn_combine: one CTA per (query head, sequence) merges the chunks
//     (rescaling by exp(m_c - max m); contiguous chunk ranges summed in
//     parallel, then added in order) and writes bf16 O, or zeros for an
//     inactive group or an empty cache.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace wide {
namespace {

constexpr int kChunk = 128;      // keys per work item
constexpr int kThreads = 128;    // 4 warps

__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&h);
}

// Warp-level bf16 tensor-core product D += A B (m16n8k16, fp32 accumulate).
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_trans(uint32_t addr, uint32_t &r0, uint32_t &r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Byte offset of 16-byte chunk c (of d) of key row r in a K or V tile as the
// TMA lays it out: 64-column halves of 128 rows x 128 B, 128-byte swizzle.
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
    return static_cast<uint32_t>((c >> 3) * (kChunk * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// One CTA per (128-key chunk, KV head, sequence).  The group's QPK query heads
// are rows 0..QPK-1 of a 16-row MMA tile (rows QPK..15 are zero).
template <int D, int QPK>
__global__ void __launch_bounds__(kThreads)
    attn_partial_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const AttnDecodeArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    constexpr int HALVES = D / 64;
    constexpr int TILE = HALVES * kChunk * 128;  // bytes of the K (or V) tile
    constexpr int NW = kThreads / 32;
    uint8_t *ks = smem;
    uint8_t *vs = smem + TILE;
    float *ps = reinterpret_cast<float *>(smem + 2 * TILE);  // [kChunk][QPK]
    uint64_t *bar = reinterpret_cast<uint64_t *>(ps + kChunk * QPK);

    // the combine kernel (a programmatic dependent) may be scheduled now; it
    // waits for this grid before it reads the partials
    griddep_launch_dependents();
    const int chunk = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int L = min(max(a.lens[b], 0), a.L_max);  // lengths outside [0, L_max] are clamped
    const int j0 = chunk * kChunk;
    if (a.mask[static_cast<size_t>(b) * a.Hk + g] == 0 || j0 >= L) return;
    const int n_keys = min(kChunk, L - j0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;  // MMA fragment coordinates

    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // rows of the [B * Hk * L_max, d] cache view; a box may run past this
        // head's keys (rows n_keys.. are never used, and V's are zeroed below)
        const int row = (b * a.Hk + g) * a.L_max + j0;
        mbar_arrive_expect_tx(bar, 2 * TILE);
#pragma unroll
        for (int hf = 0; hf < HALVES; ++hf) {
            tma_load_2d(ks + hf * kChunk * 128, &tmK, bar, hf * 64, row);
            tma_load_2d(vs + hf * kChunk * 128, &tmV, bar, hf * 64, row);
        }
    }

    // A fragments of Q (bf16 pairs; rows gid >= QPK are zero), all k-steps over d
    uint32_t qa[D / 16][2];
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
        if (gid < QPK) {
            const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
                a.Q + (static_cast<size_t>(b) * a.Hq + g * QPK + gid) * D + k * 16);
            qa[k][0] = qrow[tig];
            qa[k][1] = qrow[4 + tig];
        } else {
            qa[k][0] = qa[k][1] = 0u;
        }
    }
    int ok = 1;
    if (lane == 0) ok = mbar_wait(bar, 0, a.status);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!__syncthreads_and(ok)) {
        // the status word records the timeout; give the copies one more bounded
        // wait before the CTA's shared memory is released
        if (threadIdx.x == 0) mbar_wait(bar, 0, nullptr);
        return;
    }
    // V rows past the chunk's keys hold other data: make them exact zeros
    if (n_keys < kChunk) {
        const int n16 = (kChunk - n_keys) * 8 * HALVES;  // 16-byte chunks to clear
        for (int i = threadIdx.x; i < n16; i += kThreads) {
            const int hf = i / ((kChunk - n_keys) * 8), rem = i % ((kChunk - n_keys) * 8);
            const int r = n_keys + rem / 8, c = rem % 8;
            *reinterpret_cast<uint4 *>(vs + hf * kChunk * 128 + r * 128 + (c << 4)) = make_uint4(0, 0, 0, 0);
        }
    }

    // S = Q K^T / sqrt(d): warp w takes keys [32 w, 32 w + 32) (four 8-key tiles)
    const float scale = rsqrtf(static_cast<float>(D));
    const uint32_t ks_u = smem_u32(ks), vs_u = smem_u32(vs);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int n0 = warp * 32 + t * 8;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
            // lanes 0..7: rows n0.., d chunk 2k; lanes 8..15: same rows, chunk 2k + 1
            const int r = n0 + (lane & 7), c = 2 * k + ((lane >> 3) & 1);
            uint32_t b0, b1;
            ldsm_x2(ks_u + sw_off(r, c), b0, b1);
            mma16816(acc, qa[k][0], qa[k][1], b0, b1);
        }
        if (gid < QPK) {
            const int j = n0 + 2 * tig;
            if (j < n_keys) ps[j * QPK + gid] = acc[0] * scale;
            if (j + 1 < n_keys) ps[(j + 1) * QPK + gid] = acc[1] * scale;
        }
    }
    __syncthreads();

    // per head: chunk maximum, exp(s - m) and its sum; p = 0 past n_keys
    for (int h = warp; h < QPK; h += NW) {
        float m = -INFINITY;
        for (int j = lane; j < n_keys; j += 32) m = fmaxf(m, ps[j * QPK + h]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.f;
        for (int j = lane; j < kChunk; j += 32) {
            const float p = j < n_keys ? expf(ps[j * QPK + h] - m) : 0.f;
            ps[j * QPK + h] = p;
            l += p;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            const size_t idx = (static_cast<size_t>(b) * a.Hq + g * QPK + h) * a.n_chunks + chunk;
            a.ws_ml[2 * idx] = m;
            a.ws_ml[2 * idx + 1] = l;
        }
    }
    __syncthreads();

    // O = P V: A = P (bf16, heads x keys), B = V via transposed ldmatrix; warp
    // w owns d columns [w * D/4, (w+1) * D/4) (D/32 eight-column tiles)
    constexpr int NT = D / 32;
    float o[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
#pragma unroll
    for (int k = 0; k < kChunk / 16; ++k) {
        uint32_t a0 = 0u, a2 = 0u;
        if (gid < QPK) {
            const int j = k * 16 + 2 * tig;
            a0 = pack2(ps[j * QPK + gid], ps[(j + 1) * QPK + gid]);
            a2 = pack2(ps[(j + 8) * QPK + gid], ps[(j + 9) * QPK + gid]);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int n0 = warp * (D / 4) + t * 8;
            // lanes 0..7: key rows 16k.., lanes 8..15: rows 16k+8..; the d chunk of n0
            const int r = k * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, c = n0 >> 3;
            uint32_t b0, b1;
            ldsm_x2_trans(vs_u + sw_off(r, c), b0, b1);
            mma16816(o[t], a0, a2, b0, b1);
        }
    }
    if (gid < QPK) {
        const size_t idx = (static_cast<size_t>(b) * a.Hq + g * QPK + gid) * a.n_chunks + chunk;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int n0 = warp * (D / 4) + t * 8;
            *reinterpret_cast<float2 *>(a.ws_o + idx * D + n0 + 2 * tig) = make_float2(o[t][0], o[t][1]);
        }
    }
}

// Block-wide reductions of the combine (fixed shuffle and warp order, so the
// result does not depend on timing).  `red` holds one float per warp.
constexpr int kCombThreads = 512;

__device__ __forceinline__ float comb_block_max(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        float w = threadIdx.x < kCombThreads / 32 ? red[threadIdx.x] : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w = fmaxf(w, __shfl_xor_sync(0xffffffffu, w, o));
        if (threadIdx.x == 0) red[kCombThreads / 32] = w;
    }
    __syncthreads();
    return red[kCombThreads / 32];
}

__device__ __forceinline__ float comb_block_sum(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();  // red may still be read by comb_block_max's callers
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        float w = threadIdx.x < kCombThreads / 32 ? red[threadIdx.x] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
        if (threadIdx.x == 0) red[kCombThreads / 32] = w;
    }
    __syncthreads();
    return red[kCombThreads / 32];
}

// One CTA per (query head, sequence) merges the chunk partials: M = max_c m_c,
// w_c = exp(m_c - M), O = sum_c w_c o_c / sum_c w_c l_c.  The chunks' (m, l)
// pairs are read by one thread each, and the weighted sum of the o_c rows is
// cut into kCombThreads / D contiguous chunk ranges, each summed by D threads
// with sixteen loads in flight; the ranges' sums are then added in order.
template <int D>
__global__ void __launch_bounds__(kCombThreads)
    attn_combine_kernel(const AttnDecodeArgs a) {
    static_assert(kCombThreads % D == 0, "whole parts of D threads");
    constexpr int kParts = kCombThreads / D;
    griddep_wait();  // the chunk partials are the previous kernel's output
    __shared__ float wts[1024];  // per-chunk weights exp(m_c - M)
    __shared__ float red[kCombThreads / 32 + 1];
    __shared__ float part[kCombThreads];  // [kParts][D] sums of the chunk ranges
    const int h = blockIdx.x, b = blockIdx.y;
    const int qpk = a.Hq / a.Hk, g = h / qpk;
    const int L = min(max(a.lens[b], 0), a.L_max);
    const bool active = a.mask[static_cast<size_t>(b) * a.Hk + g] != 0 && L > 0;
    uint16_t *orow = a.O + (static_cast<size_t>(b) * a.Hq + h) * D;
    if (!active) {
        for (int e = threadIdx.x; e < D; e += kCombThreads) orow[e] = 0;
        return;
    }
    const int n_valid = (L + kChunk - 1) / kChunk;  // <= 1022 (L_max checked on the host)
    const size_t base = (static_cast<size_t>(b) * a.Hq + h) * a.n_chunks;
    // (m, l) of chunks tid and tid + kCombThreads
    float m_c[2], l_c[2];
    float mloc = -INFINITY;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int c = threadIdx.x + k * kCombThreads;
        m_c[k] = c < n_valid ? a.ws_ml[2 * (base + c)] : -INFINITY;
        l_c[k] = c < n_valid ? a.ws_ml[2 * (base + c) + 1] : 0.f;
        mloc = fmaxf(mloc, m_c[k]);
    }
    const float M = comb_block_max(mloc, red);
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int c = threadIdx.x + k * kCombThreads;
        if (c < n_valid) {
            const float w = expf(m_c[k] - M);
            wts[c] = w;
            t += w * l_c[k];
        }
    }
    const float inv = 1.f / comb_block_sum(t, red);  // also publishes wts
    // weighted sum of the o rows over this thread's chunk range
    const int p = threadIdx.x / D, e = threadIdx.x - p * D;
    const int per = (n_valid + kParts - 1) / kParts;
    const int c0 = min(n_valid, p * per), c1 = min(n_valid, c0 + per);
    const float *src = a.ws_o + (base + c0) * D + e;
    float o = 0.f;
    int c = c0;
    for (; c + 16 <= c1; c += 16, src += 16 * D) {
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = src[j * D];
#pragma unroll
        for (int j = 0; j < 16; ++j) o = fmaf(v[j], wts[c + j], o);
    }
    for (; c < c1; ++c, src += D) o = fmaf(*src, wts[c], o);
    part[threadIdx.x] = o;
    __syncthreads();
    if (threadIdx.x < D) {
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < kParts; ++q) sum += part[q * D + threadIdx.x];
        orow[threadIdx.x] = f32_to_bf16(sum * inv);
    }
}

template <int D, int QPK>
cudaError_t launch_t(const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnDecodeArgs &a,
                     cudaStream_t s) {
    const size_t smem = 1024 + 2 * (D / 64) * kChunk * 128 + kChunk * QPK * 4 + 16;
    auto kp = attn_partial_kernel<D, QPK>;
    cudaError_t e = cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kp<<<dim3(a.n_chunks, a.Hk, a.B), kThreads, smem, s>>>(tmK, tmV, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // the combine overlaps the chunk kernel's tail (programmatic dependent launch)
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.Hq, a.B);
    cfg.blockDim = dim3(kCombThreads);
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_combine_kernel<D>, a);
}

template <int D>
cudaError_t launch_d(const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnDecodeArgs &a,
                     cudaStream_t s) {
    switch (a.Hq / a.Hk) {
        case 1: return launch_t<D, 1>(tmK, tmV, a, s);
        case 2: return launch_t<D, 2>(tmK, tmV, a, s);
        case 4: return launch_t<D, 4>(tmK, tmV, a, s);
        case 8: return launch_t<D, 8>(tmK, tmV, a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int attn_decode_chunks(int L_max) { return (L_max + kChunk - 1) / kChunk; }

// Workspace: (m, l) float pairs [B, Hq, n_chunks][2], then (16-byte aligned)
// o [B, Hq, n_chunks][d] float.
size_t attn_decode_ml_bytes(int B, int Hq, int L_max) {
    const size_t n = static_cast<size_t>(B) * Hq * attn_decode_chunks(L_max);
    return (n * 2 * sizeof(float) + 15) & ~static_cast<size_t>(15);
}

size_t attn_decode_workspace_bytes(int B, int Hq, int d, int L_max) {
    const size_t n = static_cast<size_t>(B) * Hq * attn_decode_chunks(L_max);
    return attn_decode_ml_bytes(B, Hq, L_max) + n * static_cast<size_t>(d) * sizeof(float);
}

bool attn_decode_supported(int Hq, int Hk, int d, int L_max) {
    if (d != 64 && d != 128) return false;
    if (Hk < 1 || Hq % Hk) return false;
    const int qpk = Hq / Hk;
    if (qpk != 1 && qpk != 2 && qpk != 4 && qpk != 8) return false;
    return attn_decode_chunks(L_max) <= 1022;  // the combine stages the chunk weights
}

cudaError_t launch_attn_decode(const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnDecodeArgs &a,
                               cudaStream_t s) {
    if (a.d == 64) return launch_d<64>(tmK, tmV, a, s);
    if (a.d == 128) return launch_d<128>(tmK, tmV, a, s);
    return cudaErrorInvalidValue;
}

}  // namespace wide
