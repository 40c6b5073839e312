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
//   attn_partial: persistent CTAs walk the (sequence, KV head, 128-key chunk)
//     items; items of an inactive group, or past lens[b], are skipped without
//     a read.  K and V of an item arrive by two bulk copies (TMA engine) into
//     one of two shared-memory buffers, the next item's copies running while
//     the current one is computed; the
//     scores of all the group's query heads come from lane-split partial dot
//     products over eight keys at a time and a butterfly reduce-scatter; each
//     head's chunk maximum m, sum l = sum exp(s - m) and o = sum exp(s - m) v
//     go to the workspace.
//   attn_combine: one CTA per (query head, sequence) merges the chunks in
//     order (rescaling by exp(m_c - max m)) and writes bf16 O, or zeros for
//     an inactive group or an empty cache.
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

// p of key j for all QPK heads, one vector load (ps is [key][QPK]).
template <int QPK>
__device__ __forceinline__ void load_p(const float *ps, int j, float (&p)[QPK]) {
    if constexpr (QPK == 1) {
        p[0] = ps[j];
    } else if constexpr (QPK == 2) {
        const float2 v = reinterpret_cast<const float2 *>(ps)[j];
        p[0] = v.x; p[1] = v.y;
    } else {
#pragma unroll
        for (int c = 0; c < QPK / 4; ++c) {
            const float4 v = reinterpret_cast<const float4 *>(ps + j * QPK)[c];
            p[4 * c] = v.x; p[4 * c + 1] = v.y; p[4 * c + 2] = v.z; p[4 * c + 3] = v.w;
        }
    }
}

// One work item: 128 keys of one (sequence b, KV head g).  Returns false for
// items that read nothing (inactive group, or past the sequence's keys).
struct Item {
    int b, g, chunk, n_keys;
};

__device__ __forceinline__ bool item_of(const AttnDecodeArgs &a, int i, Item &it) {
    it.chunk = i % a.n_chunks;
    const int bg = i / a.n_chunks;
    it.g = bg % a.Hk;
    it.b = bg / a.Hk;
    const int L = min(max(a.lens[it.b], 0), a.L_max);  // lengths outside [0, L_max] are clamped
    const int j0 = it.chunk * kChunk;
    it.n_keys = min(kChunk, L - j0);
    return a.mask[static_cast<size_t>(it.b) * a.Hk + it.g] != 0 && j0 < L;
}

// NB = 2: persistent CTAs, the next item's copies overlap the current item's
// compute.  NB = 1: one item per CTA, several CTAs per SM overlap instead.
template <int D, int QPK, int NB>
__global__ void __launch_bounds__(kThreads)
    attn_partial_kernel(const AttnDecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int ROW = D * 2;      // bytes of a K or V row
    constexpr int BUF = 2 * kChunk * ROW;  // K then V of one item
    constexpr int E = D / 32;       // elements of d per lane in the score phase
    constexpr int NW = kThreads / 32;
    float *ps = reinterpret_cast<float *>(smem + NB * BUF);                   // [kChunk][QPK]
    float *red = ps + kChunk * QPK;                                           // [kThreads][2 QPK]
    uint64_t *bar = reinterpret_cast<uint64_t *>(red + kThreads * 2 * QPK);  // [2]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_items = a.B * a.Hk * a.n_chunks;
    const int stride = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_barrier_init();
    }
    __syncthreads();

    // every thread walks the same item sequence (the mask and lens reads hit L1)
    auto next_item = [&](int i, Item &it) {
        while (i < n_items && !item_of(a, i, it)) i += stride;
        return i;
    };
    auto issue = [&](const Item &it, int buf) {  // thread 0: K and V of `it` into buffer buf
        const size_t off = ((static_cast<size_t>(it.b) * a.Hk + it.g) * a.L_max + it.chunk * kChunk) * D;
        uint8_t *dst = smem + buf * BUF;
        const uint32_t bytes = static_cast<uint32_t>(it.n_keys * ROW);
        mbar_arrive_expect_tx(&bar[buf], 2 * bytes);
        bulk_load_1d(dst, a.K + off, bytes, &bar[buf]);
        bulk_load_1d(dst + kChunk * ROW, a.V + off, bytes, &bar[buf]);
    };

    Item cur, nxt;
    int icur = next_item(blockIdx.x, cur);
    if (threadIdx.x == 0 && icur < n_items) issue(cur, 0);
    int inxt = icur < n_items ? next_item(icur + stride, nxt) : n_items;
    int buf = 0;
    uint32_t phases = 0u;                          // bit i: parity of buffer i's next completion
    uint32_t loaded = icur < n_items ? 1u : 0u;    // bit i: copies in flight into buffer i
    bool abort = false;
    const float scale = rsqrtf(static_cast<float>(D));

    while (icur < n_items) {
        // prefetch the next item into the other buffer (freed at the end of the last iteration)
        if (NB == 2 && inxt < n_items) {
            if (threadIdx.x == 0) issue(nxt, buf ^ 1);
            loaded |= 1u << (buf ^ 1);
        }
        const uint16_t *ks = reinterpret_cast<const uint16_t *>(smem + buf * BUF);
        const uint16_t *vs = ks + kChunk * D;
        const int b = cur.b, g = cur.g, n_keys = cur.n_keys;

        // this lane's E elements of every query head of the group, scaled by 1/sqrt(d)
        float q[QPK][E];
#pragma unroll
        for (int h = 0; h < QPK; ++h) {
            const uint16_t *qrow = a.Q + (static_cast<size_t>(b) * a.Hq + g * QPK + h) * D + lane * E;
#pragma unroll
            for (int e = 0; e < E; ++e) q[h][e] = __uint_as_float(static_cast<uint32_t>(qrow[e]) << 16) * scale;
        }
        int ok = 1;
        if (lane == 0) ok = mbar_wait(&bar[buf], (phases >> buf) & 1u, a.status);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!__syncthreads_and(ok)) { abort = true; break; }
        loaded &= ~(1u << buf);
        phases ^= 1u << buf;

        // Scores, eight keys per warp step: every lane forms partial dot
        // products over its E elements for 8 keys x QPK heads, then a butterfly
        // reduce-scatter (xor 16, 8, 4 halve the key set, xor 2, 1 finish the
        // sum) leaves the full score of key (lane >> 2) & 7 in each lane quad.
        for (int jb = warp * 8; jb < n_keys; jb += NW * 8) {
            float v[8][QPK];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                float kv[E];
                const int j = min(jb + k, n_keys - 1);  // rows past n_keys are not used
                const uint16_t *krow = ks + j * D + lane * E;  // a warp reads one whole row
                if constexpr (E == 4) {
                    const uint2 w = *reinterpret_cast<const uint2 *>(krow);
                    kv[0] = __uint_as_float(w.x << 16);
                    kv[1] = __uint_as_float(w.x & 0xFFFF0000u);
                    kv[2] = __uint_as_float(w.y << 16);
                    kv[3] = __uint_as_float(w.y & 0xFFFF0000u);
                } else {
                    const uint32_t w = *reinterpret_cast<const uint32_t *>(krow);
                    kv[0] = __uint_as_float(w << 16);
                    kv[1] = __uint_as_float(w & 0xFFFF0000u);
                }
#pragma unroll
                for (int h = 0; h < QPK; ++h) {
                    float sc = 0.f;
#pragma unroll
                    for (int e = 0; e < E; ++e) sc = fmaf(q[h][e], kv[e], sc);
                    v[k][h] = sc;
                }
            }
#pragma unroll
            for (int step = 0; step < 3; ++step) {
                const int m = 16 >> step;    // 16, 8, 4
                const int half = 4 >> step;  // keys kept after this step: 4, 2, 1
                const bool upper = (lane & m) != 0;
#pragma unroll
                for (int k = 0; k < half; ++k)
#pragma unroll
                    for (int h = 0; h < QPK; ++h) {
                        const float send = upper ? v[k][h] : v[k + half][h];
                        const float keep = upper ? v[k + half][h] : v[k][h];
                        v[k][h] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                    }
            }
#pragma unroll
            for (int h = 0; h < QPK; ++h) {
                v[0][h] += __shfl_xor_sync(0xffffffffu, v[0][h], 2);
                v[0][h] += __shfl_xor_sync(0xffffffffu, v[0][h], 1);
            }
            const int j = jb + ((lane >> 2) & 7);
            if ((lane & 3) == 0 && j < n_keys) {
#pragma unroll
                for (int h = 0; h < QPK; ++h) ps[j * QPK + h] = v[0][h];
            }
        }
        __syncthreads();

        // per head: chunk maximum, exp(s - m) and its sum (warp w handles heads w, w+NW, ...)
        for (int h = warp; h < QPK; h += NW) {
            float m = -INFINITY;
            for (int j = lane; j < n_keys; j += 32) m = fmaxf(m, ps[j * QPK + h]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            float l = 0.f;
            for (int j = lane; j < n_keys; j += 32) {
                const float p = expf(ps[j * QPK + h] - m);
                ps[j * QPK + h] = p;
                l += p;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
            if (lane == 0) {
                const size_t idx = (static_cast<size_t>(b) * a.Hq + g * QPK + h) * a.n_chunks + cur.chunk;
                a.ws_ml[2 * idx] = m;
                a.ws_ml[2 * idx + 1] = l;
            }
        }
        __syncthreads();

        // o[h][e] = sum_j p[h][j] v[j][e]: a thread owns the element pair (2c, 2c+1)
        // and one of KS key slices; the slices are added through shared memory.
        constexpr int PAIRS = D / 2;
        constexpr int KS = kThreads / PAIRS;
        const int c = threadIdx.x % PAIRS, slice = threadIdx.x / PAIRS;
        const int per = (n_keys + KS - 1) / KS;
        const int jlo = slice * per, jhi = min(n_keys, jlo + per);
        float acc[QPK][2];
#pragma unroll
        for (int h = 0; h < QPK; ++h) acc[h][0] = acc[h][1] = 0.f;
        for (int j = jlo; j < jhi; ++j) {
            const uint32_t w = reinterpret_cast<const uint32_t *>(vs + j * D)[c];
            const float v0 = __uint_as_float(w << 16), v1 = __uint_as_float(w & 0xFFFF0000u);
            float p[QPK];
            load_p<QPK>(ps, j, p);
#pragma unroll
            for (int h = 0; h < QPK; ++h) {
                acc[h][0] = fmaf(p[h], v0, acc[h][0]);
                acc[h][1] = fmaf(p[h], v1, acc[h][1]);
            }
        }
        if (slice > 0) {
#pragma unroll
            for (int h = 0; h < QPK; ++h) {
                red[threadIdx.x * 2 * QPK + 2 * h] = acc[h][0];
                red[threadIdx.x * 2 * QPK + 2 * h + 1] = acc[h][1];
            }
        }
        __syncthreads();
        if (slice == 0) {
            for (int sl = 1; sl < KS; ++sl) {
                const float *r = red + (sl * PAIRS + c) * 2 * QPK;
#pragma unroll
                for (int h = 0; h < QPK; ++h) {  // slices added in order: deterministic
                    acc[h][0] += r[2 * h];
                    acc[h][1] += r[2 * h + 1];
                }
            }
#pragma unroll
            for (int h = 0; h < QPK; ++h) {
                const size_t idx = (static_cast<size_t>(b) * a.Hq + g * QPK + h) * a.n_chunks + cur.chunk;
                *reinterpret_cast<float2 *>(a.ws_o + idx * D + 2 * c) = make_float2(acc[h][0], acc[h][1]);
            }
        }
        __syncthreads();  // buffer `buf`, ps and red are free for the next item

        cur = nxt;
        icur = inxt;
        inxt = icur < n_items ? next_item(icur + stride, nxt) : n_items;
        if constexpr (NB == 2) {
            buf ^= 1;
        } else if (icur < n_items) {  // single buffer: load the next item only now
            if (threadIdx.x == 0) issue(cur, 0);
            loaded |= 1u;
        }
    }
    if (abort && threadIdx.x == 0) {
        // the status word records the timeout; give copies still in flight one
        // more bounded wait before the CTA's shared memory is released
        for (int i = 0; i < 2; ++i)
            if ((loaded >> i) & 1u) mbar_wait(&bar[i], (phases >> i) & 1u, nullptr);
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads)
    attn_combine_kernel(const AttnDecodeArgs a) {
    __shared__ float wts[1024];  // per-chunk weights exp(m_c - M) / sum
    const int h = blockIdx.x, b = blockIdx.y;
    const int qpk = a.Hq / a.Hk, g = h / qpk;
    const int L = min(max(a.lens[b], 0), a.L_max);
    const bool active = a.mask[static_cast<size_t>(b) * a.Hk + g] != 0 && L > 0;
    uint16_t *orow = a.O + (static_cast<size_t>(b) * a.Hq + h) * D;
    if (!active) {
        for (int e = threadIdx.x; e < D; e += kThreads) orow[e] = 0;
        return;
    }
    const int n_valid = (L + kChunk - 1) / kChunk;
    const size_t base = (static_cast<size_t>(b) * a.Hq + h) * a.n_chunks;
    // maximum and normaliser over the chunks (one warp, chunks in ascending order)
    if (threadIdx.x < 32) {
        float M = -INFINITY;
        for (int c = threadIdx.x; c < n_valid; c += 32) M = fmaxf(M, a.ws_ml[2 * (base + c)]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float wsum = 0.f;
        for (int c0 = 0; c0 < n_valid; c0 += 32) {
            const int c = c0 + threadIdx.x;
            const float w = c < n_valid ? expf(a.ws_ml[2 * (base + c)] - M) : 0.f;
            if (c < n_valid) wts[c % 1024] = w;
            float t = c < n_valid ? w * a.ws_ml[2 * (base + c) + 1] : 0.f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
            wsum += t;
        }
        if (threadIdx.x == 0) wts[1023] = 1.f / wsum;  // n_valid <= 1022 (L_max checked on the host)
    }
    __syncthreads();
    const float inv = wts[1023];
    for (int e = threadIdx.x; e < D; e += kThreads) {
        float o = 0.f;
#pragma unroll 8
        for (int c = 0; c < n_valid; ++c) o = fmaf(a.ws_o[(base + c) * D + e], wts[c], o);
        orow[e] = f32_to_bf16(o * inv);
    }
}

template <int D, int QPK>
cudaError_t launch_t(const AttnDecodeArgs &a, int num_sms, cudaStream_t s) {
    // one K+V buffer per CTA, one item per CTA (several CTAs per SM), plus the
    // chunk's p values and the slice reduction area
    constexpr int NB = 1;
    (void)num_sms;
    const size_t smem = NB * (2 * kChunk * D * 2) + kChunk * QPK * 4 + kThreads * 2 * QPK * 4 + 2 * 8;
    auto kp = attn_partial_kernel<D, QPK, NB>;
    cudaError_t e = cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const long long items = static_cast<long long>(a.B) * a.Hk * a.n_chunks;
    if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
    kp<<<static_cast<int>(items), kThreads, smem, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    attn_combine_kernel<D><<<dim3(a.Hq, a.B), kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const AttnDecodeArgs &a, int num_sms, cudaStream_t s) {
    switch (a.Hq / a.Hk) {
        case 1: return launch_t<D, 1>(a, num_sms, s);
        case 2: return launch_t<D, 2>(a, num_sms, s);
        case 4: return launch_t<D, 4>(a, num_sms, s);
        case 8: return launch_t<D, 8>(a, num_sms, s);
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

cudaError_t launch_attn_decode(const AttnDecodeArgs &a, int num_sms, cudaStream_t s) {
    if (a.d == 64) return launch_d<64>(a, num_sms, s);
    if (a.d == 128) return launch_d<128>(a, num_sms, s);
    return cudaErrorInvalidValue;
}

}  // namespace wide
