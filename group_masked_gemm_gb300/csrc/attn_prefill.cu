// attn_prefill.cu -- routed causal prefill attention (WIDE, App. B
// "Implementation of Attention", prefill, Algorithm 4; GQA-aligned routing
// groups of Sec. 3.1 Eq. 2) on the warp-level tensor-core instruction, the
// kernel for head dim 64 (head dim 128 runs on tcgen05, attn_prefill_tc.cu).
//
// Query head h of sequence b reads KV head g = h / (Hq/Hk), which is also its
// routing group.  The stable partition of the group's mask column (perm,
// counts) lists the active tokens in ascending position, so a CTA owns 64
// consecutive entries of that list -- a tile of gathered query rows whose
// largest position bounds the causal key range (query-tile admission and the
// shortened KV stream of Algorithm 4).  K and V stay dense.
//
// Per CTA (4 warps, 16 query rows each):
//   - the 64 query rows are gathered with cp.async into a 128-byte-swizzled
//     tile and read into MMA fragments with ldmatrix;
//   - 64-key tiles of K and V arrive by TMA (128-byte swizzle), two stages;
//   - S = Q K^T and O += P V run on the warp-level tensor-core instruction
//     (mma.sync m16n8k16, bf16 in, fp32 accumulate); the online softmax keeps
//     a running maximum and sum per row in fp32, and P is reused from the S
//     fragments as bf16 A fragments;
//   - only key tiles that reach past the smallest query position of the tile
//     apply the element-wise causal cut;
//   - rows are scattered back to O[b, token, h, :]; the tile's inactive rows
//     (entries past counts) and every row of a fully inactive tile are
//     written as zeros, so each row of O is written exactly once.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace wide {
namespace {

constexpr int BQ = 64;       // gathered query rows per CTA
constexpr int BKV = 64;      // keys per K/V tile
constexpr int kThreads = 128;
constexpr int kStages = 2;

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
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

// Byte offset of 16-byte chunk c of row r in a tile of `rows` rows stored as
// 64-column halves of rows x 128 B with the 128-byte swizzle (the TMA layout).
__device__ __forceinline__ uint32_t sw_off(int rows, int r, int c) {
    return static_cast<uint32_t>((c >> 3) * (rows * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kThreads)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const AttnPrefillArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    constexpr int HALVES = D / 64;
    constexpr int QTILE = HALVES * BQ * 128;   // bytes of the gathered Q tile
    constexpr int KVTILE = HALVES * BKV * 128; // bytes of one K (or V) tile
    uint8_t *qs = smem;
    uint8_t *kvs = smem + QTILE;               // [stage][K tile, V tile]
    int *toks = reinterpret_cast<int *>(kvs + kStages * 2 * KVTILE);  // [BQ]
    uint64_t *bar = reinterpret_cast<uint64_t *>(toks + BQ);         // [kStages]

    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int T = a.T, qpk = a.Hq / a.Hk, g = h / qpk;
    const int cnt = a.counts[b * a.Hk + g];
    const int m0 = qt * BQ;
    const int32_t *pg = a.perm + (static_cast<size_t>(b) * a.Hk + g) * T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    auto orow = [&](int tok) { return a.O + ((static_cast<size_t>(b) * T + tok) * a.Hq + h) * D; };

    // rows m0.. of the list that are not admitted: inactive tokens, written as zeros
    const int nvalid = max(0, min(BQ, cnt - m0));
    for (int i = threadIdx.x; i < (BQ - nvalid) * (D / 8); i += kThreads) {
        const int r = nvalid + i / (D / 8), c = i % (D / 8);
        if (m0 + r < T) *reinterpret_cast<uint4 *>(orow(pg[m0 + r]) + 8 * c) = make_uint4(0, 0, 0, 0);
    }
    if (nvalid == 0) return;

    if (threadIdx.x < BQ) toks[threadIdx.x] = threadIdx.x < nvalid ? pg[m0 + threadIdx.x] : -1;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1);
        fence_barrier_init();
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
    }
    __syncthreads();
    const int max_pos = toks[nvalid - 1], min_pos = toks[0];  // ascending (stable partition)
    const int n_kv = a.causal ? max_pos / BKV + 1 : (T + BKV - 1) / BKV;
    const int kv_row0 = (b * a.Hk + g) * T;  // row of key 0 in the [B * Hk * T, d] view

    // thread 0: bit s of issued_any = stage s has been loaded at least once,
    // bit s of issued_par = parity of the last load into stage s
    uint32_t issued_any = 0u, issued_par = 0u;
    auto issue = [&](int kt, int s) {  // thread 0: K and V tile kt into stage s
        if (issued_any & (1u << s)) issued_par ^= 1u << s;
        issued_any |= 1u << s;
        uint8_t *kd = kvs + s * 2 * KVTILE;
        mbar_arrive_expect_tx(&bar[s], 2 * KVTILE);
#pragma unroll
        for (int hf = 0; hf < HALVES; ++hf) {
            tma_load_2d(kd + hf * BKV * 128, &tmK, &bar[s], hf * 64, kv_row0 + kt * BKV);
            tma_load_2d(kd + KVTILE + hf * BKV * 128, &tmV, &bar[s], hf * 64, kv_row0 + kt * BKV);
        }
    };
    if (threadIdx.x == 0) {
        issue(0, 0);
        if (n_kv > 1) issue(1, 1);
    }

    // gather the admitted query rows (zeros for the rest) into the swizzled Q tile
    const uint32_t qs_u = smem_u32(qs);
    for (int i = threadIdx.x; i < BQ * (D / 8); i += kThreads) {
        const int r = i / (D / 8), c = i % (D / 8);
        const uint32_t dst = qs_u + sw_off(BQ, r, c);
        const int tok = toks[r];
        if (tok >= 0) {
            cp_async16(dst, a.Q + ((static_cast<size_t>(b) * T + tok) * a.Hq + h) * D + 8 * c);
        } else {
            *reinterpret_cast<uint4 *>(qs + sw_off(BQ, r, c)) = make_uint4(0, 0, 0, 0);
        }
    }
    cp_async_wait_all();
    __syncthreads();

    // this warp's 16 query rows as A fragments, all k-steps over d
    uint32_t qa[D / 16][4];
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
        // lanes 0-7 rows 0-7 / 8-15 rows 8-15 of chunk 2k; lanes 16-31 the same rows of chunk 2k+1
        const int r = warp * 16 + (lane & 15), c = 2 * k + (lane >> 4);
        ldsm_x4(qs_u + sw_off(BQ, r, c), qa[k]);
    }
    // positions of this thread's two rows (rows past nvalid behave like the last row)
    const int r0 = warp * 16 + gid, r1 = r0 + 8;
    const int qpos0 = r0 < nvalid ? toks[r0] : max_pos, qpos1 = r1 < nvalid ? toks[r1] : max_pos;

    const float sl2 = rsqrtf(static_cast<float>(D)) * 1.4426950408889634f;  // 1/sqrt(d) * log2(e)
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int t = 0; t < D / 8; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
    bool ok = true;

    for (int kt = 0; kt < n_kv; ++kt) {
        const int s = kt % kStages;
        int w = 1;
        if (lane == 0) w = mbar_wait(&bar[s], (kt / kStages) & 1, a.status);
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!__syncthreads_and(w)) { ok = false; break; }
        const uint32_t ks_u = smem_u32(kvs + s * 2 * KVTILE), vs_u = ks_u + KVTILE;
        const int k0 = kt * BKV;
        if (k0 + BKV > T) {
            // the tile runs past this head's keys: its V rows there hold other data
            // (P is 0 for them, but 0 * NaN is not 0), so make them exact zeros
            uint8_t *vt = kvs + s * 2 * KVTILE + KVTILE;
            const int first = T - k0;
            for (int i = threadIdx.x; i < (BKV - first) * 8 * HALVES; i += kThreads) {
                const int hf = i / ((BKV - first) * 8), rem = i % ((BKV - first) * 8);
                *reinterpret_cast<uint4 *>(vt + hf * BKV * 128 + (first + rem / 8) * 128 + ((rem % 8) << 4)) =
                    make_uint4(0, 0, 0, 0);
            }
            __syncthreads();
        }

        // S = Q K^T for 16 rows x 64 keys
        float sc[BKV / 8][4];
#pragma unroll
        for (int n = 0; n < BKV / 8; ++n) {
            sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const int r = n * 8 + (lane & 7), c = 2 * k + ((lane >> 3) & 1);
                uint32_t b0, b1;
                ldsm_x2(ks_u + sw_off(BKV, r, c), b0, b1);
                mma16816(sc[n], qa[k], b0, b1);
            }
        }
        // scale to log2 units; causal cut and keys past T (a tile may run into
        // the next head's rows) become -inf
        const bool cut = (a.causal && k0 + BKV - 1 > min_pos) || k0 + BKV > T;
#pragma unroll
        for (int n = 0; n < BKV / 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float v = sc[n][e] * sl2;
                if (cut) {
                    const int kpos = k0 + n * 8 + 2 * tig + (e & 1);
                    const int qpos = e < 2 ? qpos0 : qpos1;
                    if (kpos >= T || (a.causal && kpos > qpos)) v = -INFINITY;
                }
                sc[n][e] = v;
            }
        // online softmax over the two rows this thread holds (a row lives in a lane quad)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            float mx = -INFINITY;
#pragma unroll
            for (int n = 0; n < BKV / 8; ++n) mx = fmaxf(mx, fmaxf(sc[n][2 * rr], sc[n][2 * rr + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_new = fmaxf(m_run[rr], mx);
            const float alpha = exp2f(m_run[rr] - m_new);  // 0 on the first tile
            float sum = 0.f;
#pragma unroll
            for (int n = 0; n < BKV / 8; ++n) {
                const float p0 = exp2f(sc[n][2 * rr] - m_new), p1 = exp2f(sc[n][2 * rr + 1] - m_new);
                sc[n][2 * rr] = p0;
                sc[n][2 * rr + 1] = p1;
                sum += p0 + p1;
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            l_run[rr] = l_run[rr] * alpha + sum;
            m_run[rr] = m_new;
#pragma unroll
            for (int t = 0; t < D / 8; ++t) {
                o[t][2 * rr] *= alpha;
                o[t][2 * rr + 1] *= alpha;
            }
        }
        // O += P V: P from the S fragments (bf16), V through transposed ldmatrix
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk) {
            const uint32_t pa[4] = {pack2(sc[2 * kk][0], sc[2 * kk][1]), pack2(sc[2 * kk][2], sc[2 * kk][3]),
                                    pack2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]),
                                    pack2(sc[2 * kk + 1][2], sc[2 * kk + 1][3])};
#pragma unroll
            for (int t = 0; t < D / 8; ++t) {
                const int r = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, c = t;
                uint32_t b0, b1;
                ldsm_x2_trans(vs_u + sw_off(BKV, r, c), b0, b1);
                mma16816(o[t], pa, b0, b1);
            }
        }
        __syncthreads();  // every warp is done with stage s
        if (threadIdx.x == 0 && kt + kStages < n_kv) issue(kt + kStages, s);
    }
    if (!ok) {
        // the status word records the timeout; wait (bounded) for copies in flight
        if (threadIdx.x == 0)
            for (int st = 0; st < kStages; ++st)
                if (issued_any & (1u << st)) mbar_wait(&bar[st], (issued_par >> st) & 1u, nullptr);
        return;
    }

    // normalise and scatter the admitted rows back to their tokens
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int r = rr == 0 ? r0 : r1;
        if (r >= nvalid) continue;
        const float inv = 1.f / l_run[rr];
        uint16_t *dst = orow(toks[r]);
#pragma unroll
        for (int t = 0; t < D / 8; ++t)
            *reinterpret_cast<uint32_t *>(dst + t * 8 + 2 * tig) = pack2(o[t][2 * rr] * inv, o[t][2 * rr + 1] * inv);
    }
}

template <int D>
cudaError_t launch_t(const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnPrefillArgs &a, cudaStream_t s) {
    const size_t smem = 1024 + (D / 64) * (BQ + kStages * 2 * BKV) * 128 + BQ * 4 + kStages * 8;
    auto k = attn_prefill_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    k<<<dim3((a.T + BQ - 1) / BQ, a.Hq, a.B), kThreads, smem, s>>>(tmK, tmV, a);
    return cudaGetLastError();
}

}  // namespace

bool attn_prefill_supported(int Hq, int Hk, int d) {
    return (d == 64 || d == 128) && Hk >= 1 && Hq % Hk == 0 && Hq / Hk <= 64;
}

cudaError_t launch_attn_prefill(const CUtensorMap &tmK, const CUtensorMap &tmV, const AttnPrefillArgs &a,
                                cudaStream_t s) {
    if (a.d == 64) return launch_t<64>(tmK, tmV, a, s);
    if (a.d == 128) return launch_t<128>(tmK, tmV, a, s);
    return cudaErrorInvalidValue;
}

}  // namespace wide
