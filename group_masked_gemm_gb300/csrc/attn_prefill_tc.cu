// attn_prefill_tc.cu -- routed causal prefill attention on the 5th-generation
// tensor cores (WIDE, App. B "Implementation of Attention", prefill,
// Algorithm 4; GQA-aligned routing groups of Sec. 3.1 Eq. 2), head dim 128.
//
// The work split is the one of attn_prefill.cu: query head h of sequence b
// reads KV head g = h / (Hq/Hk), its routing group; the stable partition of
// the group's mask column lists the active tokens in ascending position, and
// a CTA owns 128 consecutive entries of that list.  The tile's largest
// position bounds the causal key range; K and V stay dense.
//
// Two CTAs share an SM (about 100 KB of shared memory and 256 TMEM columns
// each), so one CTA's softmax runs while the other's MMAs do.  Per CTA
// (7 warps):
//   warp 0      TMA producer of the 64-key K tiles (128-byte swizzle), two
//               stages, each released as soon as its S product is done;
//   warp 6      TMA producer of the 64-key V tiles, one buffer, released by
//               its P V product;
//   warp 1      TMEM owner and MMA issuer (one thread):
//                 S_j = Q K_j^T  (M = 128 queries, N = 64 keys, K = 128 dims)
//                 into one of two TMEM S buffers, then
//                 O  += P_{j-1} V_{j-1} (A = P from shared memory, B = V read
//                 MN-major straight from its TMA tile) into the TMEM O;
//   warps 2..5  softmax, one query row per thread (its TMEM lane): gather the
//               Q rows (cp.async, swizzled), then per key tile load the S row,
//               apply scale, causal cut and keys past T, keep the running max
//               and sum, write P (bf16) to shared memory, and rescale the O
//               row in TMEM only when the running max grows by more than
//               2^8 (P is formed against the running max, so a stale max is
//               exact after the final division); finally O / l is scattered
//               to O[b, token, h, :].
// Rows of the list past counts (and every row of a tile with none) are
// written as zeros, so each row of O is written exactly once.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace wide {
namespace {

constexpr int D = 128;                       // head dim
constexpr int BQ = 128;                      // gathered query rows per CTA
constexpr int BKV = 64;                      // keys per tile
constexpr int kThreadsTc = 224;              // 7 warps
constexpr int QHALF = BQ * 128;              // 64-dim half of the Q tile: 128 rows x 128 B
constexpr int QTILE = 2 * QHALF;
constexpr int KVHALF = BKV * 128;            // 64-dim half of a K or V tile
constexpr int KVTILE = 2 * KVHALF;
constexpr int PTILE = BQ * 128;              // P: 128 rows x 64 keys (one swizzled half)
constexpr int kQOff = 0;
constexpr int kKOff = QTILE;                 // [stage] K tiles
constexpr int kVOff = kKOff + 2 * KVTILE;    // the V tile
constexpr int kPOff = kVOff + KVTILE;
constexpr int kTokOff = kPOff + PTILE;
constexpr int kBarOff = kTokOff + BQ * 4;
constexpr int kNumBars = 14;
constexpr int kSmemBytes = 1024 + kBarOff + kNumBars * 8 + 16;
constexpr int kTmemCols = 256;               // S0 [0,64), S1 [64,128), O [128,256)
constexpr int kOCol = 2 * BKV;
constexpr float kRescaleSlack = 8.0f;        // log2 units a stale running max may lag

constexpr uint32_t kIdescS = idesc_bf16_f32(BQ, BKV);
// O += P V: B (V, N = dims, K = keys) is MN-major -- bit 16 of the descriptor
constexpr uint32_t kIdescPV = idesc_bf16_f32(BQ, D) | (1u << 16);

// Byte offset of 16-byte chunk c (of 16) of row r in a tile of 64-column
// halves `half` bytes apart, 128-byte swizzle (the TMA layout).
__device__ __forceinline__ uint32_t swz(int half, int r, int c) {
    return static_cast<uint32_t>((c >> 3) * half + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// 2^x on the special-function unit, denormal results flushed to zero (the
// PTX ex2.approx.ftz instruction, relative error about 2^-22: far below the
// bf16 rounding of P that follows).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction (the three-input form of PTX max.f32).
__device__ __forceinline__ float max3(float a, float b, float c) {
    float y;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
    return y;
}

// Shared-memory descriptor of an MN-major operand in the 128-byte swizzle:
// 64-element rows of the contiguous (MN) dimension, one row per K index,
// 8-row atoms 1024 B apart along K, the two 64-element MN halves `half` apart.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t smem_addr, uint32_t half) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);  // start address
    d |= static_cast<uint64_t>(half >> 4) << 16;               // leading offset: next MN half
    d |= static_cast<uint64_t>(1024 >> 4) << 32;               // stride offset: next 8 K rows
    d |= static_cast<uint64_t>(1) << 46;                       // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                       // 128-byte swizzle
    return d;
}

__global__ void __launch_bounds__(kThreadsTc, 2)
    attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                           const AttnPrefillArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    int *toks = reinterpret_cast<int *>(smem + kTokOff);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kBarOff);
    uint64_t *kfull = bars, *kempty = bars + 2, *vfull = bars + 4, *vempty = bars + 5;
    uint64_t *sfull = bars + 6, *sempty = bars + 8;
    uint64_t *pfull = bars + 10, *pvdone = bars + 11, *qready = bars + 12, *final_bar = bars + 13;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + kNumBars);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);

    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int T = a.T, qpk = a.Hq / a.Hk, g = h / qpk;
    const int cnt = a.counts[b * a.Hk + g];
    const int m0 = qt * BQ;
    const int32_t *pg = a.perm + (static_cast<size_t>(b) * a.Hk + g) * T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto orow = [&](int tok) { return a.O + ((static_cast<size_t>(b) * T + tok) * a.Hq + h) * D; };

    // rows m0.. of the list that are not admitted: inactive tokens, written as zeros
    const int nvalid = max(0, min(BQ, cnt - m0));
    for (int i = threadIdx.x; i < (BQ - nvalid) * (D / 8); i += kThreadsTc) {
        const int r = nvalid + i / (D / 8), c = i % (D / 8);
        if (m0 + r < T) *reinterpret_cast<uint4 *>(orow(pg[m0 + r]) + 8 * c) = make_uint4(0, 0, 0, 0);
    }
    if (nvalid == 0) return;

    if (threadIdx.x < BQ) toks[threadIdx.x] = threadIdx.x < nvalid ? pg[m0 + threadIdx.x] : -1;
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&kfull[s], 1);
            mbar_init(&kempty[s], 1);
            mbar_init(&sfull[s], 1);
            mbar_init(&sempty[s], 4);
        }
        mbar_init(vfull, 1);
        mbar_init(vempty, 1);
        mbar_init(pfull, 4);
        mbar_init(pvdone, 1);
        mbar_init(qready, 4);
        mbar_init(final_bar, 1);
        *s_abort = 0;
        fence_barrier_init();
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const int max_pos = toks[nvalid - 1], min_pos = toks[0];  // ascending (stable partition)
    const int n_kv = a.causal ? max_pos / BKV + 1 : (T + BKV - 1) / BKV;
    const int kv_row0 = (b * a.Hk + g) * T;  // row of key 0 in the [B * Hk * T, d] view
    const uint32_t sbase = smem_u32(smem);

    if (warp == 0 || warp == 6) {
        // ===================== TMA producers: K (warp 0), V (warp 6) =====================
        if (lane == 0) {
            const bool is_k = warp == 0;
            const CUtensorMap *tm = is_k ? &tmK : &tmV;
            int issued = 0;
            for (int j = 0; j < n_kv && !*s_abort; ++j) {
                uint64_t *full = is_k ? &kfull[j & 1] : vfull;
                uint8_t *dst = is_k ? smem + kKOff + (j & 1) * KVTILE : smem + kVOff;
                bool ok = true;
                if (is_k && j >= 2) ok = mbar_wait(&kempty[j & 1], ((j >> 1) - 1) & 1, a.status);
                if (!is_k && j >= 1) ok = mbar_wait(vempty, (j - 1) & 1, a.status);
                if (!ok) { *s_abort = 1; break; }
                const int row = kv_row0 + j * BKV;
                mbar_arrive_expect_tx(full, KVTILE);
                tma_load_2d(dst, tm, full, 0, row);
                tma_load_2d(dst + KVHALF, tm, full, 64, row);
                issued = j + 1;
            }
            // copies in flight must land before the CTA exits
            if (is_k) {
                for (int j = issued - 2 > 0 ? issued - 2 : 0; j < issued; ++j)
                    mbar_wait(&kfull[j & 1], (j >> 1) & 1, nullptr);
            } else if (issued > 0) {
                mbar_wait(vfull, (issued - 1) & 1, nullptr);
            }
        }
    } else if (warp == 1) {
        // ============================ MMA issuer ============================
        if (lane == 0) {
            bool ok = mbar_wait(qready, 0, a.status);
            for (int j = 0; ok && j <= n_kv && !*s_abort; ++j) {
                if (j < n_kv) {  // S_j = Q K_j^T
                    const int s = j & 1;
                    if (!mbar_wait(&kfull[s], (j >> 1) & 1, a.status)) { ok = false; break; }
                    if (j >= 2 && !mbar_wait(&sempty[s], ((j >> 1) - 1) & 1, a.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t q0 = sbase + kQOff, k0 = sbase + kKOff + s * KVTILE;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_bf16(tmem + s * BKV, sw128_kmajor_desc(q0 + (kk >> 2) * QHALF + (kk & 3) * 32),
                                 sw128_kmajor_desc(k0 + (kk >> 2) * KVHALF + (kk & 3) * 32), kIdescS,
                                 kk > 0 ? 1u : 0u);
                    mma_commit(&sfull[s]);
                    mma_commit(&kempty[s]);  // the K tile is no longer needed
                }
                if (j >= 1) {  // O += P_{j-1} V_{j-1}
                    const int jj = j - 1;
                    if (!mbar_wait(vfull, jj & 1, a.status)) { ok = false; break; }
                    if (!mbar_wait(pfull, jj & 1, a.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t p0 = sbase + kPOff, v0 = sbase + kVOff;
#pragma unroll
                    for (int kk = 0; kk < BKV / 16; ++kk)
                        mma_bf16(tmem + kOCol, sw128_kmajor_desc(p0 + kk * 32),
                                 sw128_mnmajor_desc(v0 + kk * 2048, KVHALF), kIdescPV,
                                 (jj > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(pvdone);
                    mma_commit(vempty);
                }
            }
            if (!ok) *s_abort = 1;
            // every MMA issued must complete before TMEM is released
            mma_commit(final_bar);
            mbar_wait(final_bar, 0, nullptr);
        }
    } else {
        // ============================ softmax warps ============================
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        // gather the admitted query rows (zeros for the rest) into the swizzled Q tile
        {
            const int tok = toks[row];
            for (int c = 0; c < D / 8; ++c) {
                const uint32_t dst = sbase + kQOff + swz(QHALF, row, c);
                if (tok >= 0)
                    cp_async16(dst, a.Q + ((static_cast<size_t>(b) * T + tok) * a.Hq + h) * D + 8 * c);
                else
                    *reinterpret_cast<uint4 *>(smem + kQOff + swz(QHALF, row, c)) = make_uint4(0, 0, 0, 0);
            }
            cp_async_wait_all();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(qready);
        }
        const int qpos = row < nvalid ? toks[row] : max_pos;  // rows past nvalid: like the last
        const float sl2 = rsqrtf(static_cast<float>(D)) * 1.4426950408889634f;  // log2(e) / sqrt(d)
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int s = j & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&sfull[s], (j >> 1) & 1, a.status))) { ok = false; break; }
            tc_fence_after();
            float v[BKV];
            {
                uint32_t r[32];
#pragma unroll
                for (int c = 0; c < BKV / 32; ++c) {
                    tmem_ld32(lane_addr + s * BKV + c * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[c * 32 + e] = __uint_as_float(r[e]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sempty[s]);  // S_j is in registers
            const int k0 = j * BKV;
            const bool cut = (a.causal && k0 + BKV - 1 > min_pos) || k0 + BKV > T;
            // raw scores; the cut ones become -inf, and the row maximum (the
            // scale is positive) runs in 2 chains of three-input maxima
            if (cut) {
#pragma unroll
                for (int e = 0; e < BKV; ++e) {
                    const int kpos = k0 + e;
                    if (kpos >= T || (a.causal && kpos > qpos)) v[e] = -INFINITY;
                }
            }
            float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
            for (int e = 0; e < BKV; e += 4) {
                mxa = max3(mxa, v[e], v[e + 1]);
                mxb = max3(mxb, v[e + 2], v[e + 3]);
            }
            const float mx = fmaxf(mxa, mxb) * sl2;
            // the running maximum; a warp rescales when any of its rows grew by
            // more than the slack (then every lane moves to its new maximum)
            const float m_new = fmaxf(m_run, mx);
            float alpha = 1.f;
            bool rescale = false;
            if (j == 0) {
                m_run = m_new;
            } else if (__any_sync(0xffffffffu, m_new > m_run + kRescaleSlack)) {
                alpha = ex2(m_run - m_new);
                m_run = m_new;
                rescale = true;
            }
            // P = exp2(x - m_run) in registers, x the scaled score: this overlaps
            // the tensor cores' P_{j-1} V_{j-1}
            float sum4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int e = 0; e < BKV; ++e) {
                v[e] = ex2(fmaf(v[e], sl2, -m_run));  // exp2(score * log2(e) / sqrt(d) - max)
                sum4[e & 3] += v[e];
            }
            const float sum = (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
            // P_{j-1} has been multiplied (the P buffer is free, O is settled)
            if (j > 0 && !__all_sync(0xffffffffu, mbar_wait(pvdone, (j - 1) & 1, a.status))) { ok = false; break; }
            tc_fence_after();
            if (rescale) {
                l_run *= alpha;
                uint32_t r[32];
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    tmem_ld32(lane_addr + kOCol + c * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                    tmem_st32(lane_addr + kOCol + c * 32, r);
                }
                tmem_st_wait();
            }
            if (k0 + BKV > T) {
                // the tile runs past this head's keys: its V rows there hold other
                // data (P is 0 for them, but 0 * NaN is not 0), so zero them
                if (!__all_sync(0xffffffffu, mbar_wait(vfull, j & 1, a.status))) { ok = false; break; }
                uint8_t *vt = smem + kVOff;
                const int first = T - k0;
                for (int i = row; i < (BKV - first) * 16; i += BQ) {
                    const int rr = first + i / 16, c = i % 16;
                    *reinterpret_cast<uint4 *>(vt + swz(KVHALF, rr, c)) = make_uint4(0, 0, 0, 0);
                }
            }
            // P as bf16 into the swizzled P tile (row = this thread)
            uint8_t *pt = smem + kPOff;
#pragma unroll
            for (int c = 0; c < BKV / 8; ++c)
                *reinterpret_cast<uint4 *>(pt + swz(PTILE, row, c)) =
                    make_uint4(pack_bf16x2(v[8 * c], v[8 * c + 1]), pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                               pack_bf16x2(v[8 * c + 4], v[8 * c + 5]), pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
            l_run += sum;
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pfull);
        }
        if (ok && !__all_sync(0xffffffffu, mbar_wait(pvdone, (n_kv - 1) & 1, a.status))) ok = false;
        if (ok) {
            tc_fence_after();
            // normalise and scatter the admitted rows back to their tokens
            const float inv = 1.f / l_run;
            uint16_t *dst = row < nvalid ? orow(toks[row]) : nullptr;
            uint32_t r[32];
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                tmem_ld32(lane_addr + kOCol + c * 32, r);
                tmem_ld_wait();
                if (dst != nullptr) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4 *>(dst + c * 32 + 8 * q) = make_uint4(
                            pack_bf16x2(__uint_as_float(r[8 * q]) * inv, __uint_as_float(r[8 * q + 1]) * inv),
                            pack_bf16x2(__uint_as_float(r[8 * q + 2]) * inv, __uint_as_float(r[8 * q + 3]) * inv),
                            pack_bf16x2(__uint_as_float(r[8 * q + 4]) * inv, __uint_as_float(r[8 * q + 5]) * inv),
                            pack_bf16x2(__uint_as_float(r[8 * q + 6]) * inv, __uint_as_float(r[8 * q + 7]) * inv));
                }
            }
        } else {
            *s_abort = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

bool attn_prefill_tc_supported(int d) { return d == D; }

cudaError_t launch_attn_prefill_tc(const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnPrefillArgs &a,
                                   cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(attn_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    // two CTAs per SM: prefer the largest shared-memory carve-out
    e = cudaFuncSetAttribute(attn_prefill_tc_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    attn_prefill_tc_kernel<<<dim3((a.T + BQ - 1) / BQ, a.Hq, a.B), kThreadsTc, kSmemBytes, s>>>(tmK, tmV, a);
    return cudaGetLastError();
}

}  // namespace wide
