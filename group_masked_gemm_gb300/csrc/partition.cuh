// partition.cuh -- the per-group stable partition of a mask (WIDE, Sec. 3.3
// Eq. 7; App. B Algorithm 1) from per-tile ballots, shared by the one-launch
// router + reorder and the cooperative reorder kernel.
//
// Tokens come in tiles of 128 (four 32-token warps' worth).  A first phase,
// in the calling kernel, stores for every (tile, group) the four 32-bit
// ballots of the tile's active tokens.  Then, in one cooperative launch:
//   - partition_scan: group g's per-tile active counts are scanned (tiles in
//     ascending order) into tile offsets and counts[g];
//   - partition_place: a token that is active in g goes to
//     offset[tile][g] + its rank among the tile's active tokens, an inactive
//     one to counts[g] + (inactive tokens before it) -- the stable partition.
// Grid barriers between the phases are bounded waits on a counter.
#pragma once

#include "common.cuh"

namespace wide {

constexpr int kPartTile = 128;  // tokens per ballot tile

// Workspace: barrier counter (16 bytes), ballots [tiles][ng][4] uint32,
// tile offsets [tiles][ng] int32.
inline size_t partition_workspace_bytes(int T, int n_groups) {
    const size_t tiles = (static_cast<size_t>(T) + kPartTile - 1) / kPartTile;
    return 16 + tiles * n_groups * (16 + 4);
}

struct PartitionWs {
    unsigned *ctr;
    uint32_t *bal;
    int32_t *off;
};

__device__ __forceinline__ PartitionWs partition_ws(uint32_t *ws, int n_tiles, int ng) {
    PartitionWs w;
    w.ctr = ws;
    w.bal = ws + 4;
    w.off = reinterpret_cast<int32_t *>(ws + 4 + static_cast<size_t>(n_tiles) * ng * 4);
    return w;
}

// Exclusive scan of v over the block; *total receives the block sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_sums, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += y;
    }
    if (lane == 31) warp_sums[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        const int w = lane < nw ? warp_sums[lane] : 0;
        int winc = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, winc, d);
            if (lane >= d) winc += y;
        }
        warp_sums[lane] = winc - w;
        if (lane == 31) *total = winc;
    }
    __syncthreads();
    const int out = warp_sums[warp] + inc - v;
    __syncthreads();
    return out;
}

// Every CTA of a cooperative launch arrives; returns once `target` arrivals
// have been counted (or false after kWaitLimitNs, recording the timeout).
// Writes before the barrier are visible to every CTA after it.
__device__ __forceinline__ bool grid_barrier(unsigned *ctr, unsigned target, int *status,
                                             volatile int *s_ok) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(ctr, 1u);
        int ok = 1;
        const unsigned long long t0 = globaltimer();
        while (*reinterpret_cast<volatile unsigned *>(ctr) < target) {
            __nanosleep(64);
            if (globaltimer() - t0 > kWaitLimitNs) {
                if (status) atomicCAS(status, 0, kStatusTimeout);
                ok = 0;
                break;
            }
        }
        __threadfence();
        *s_ok = ok;
    }
    __syncthreads();
    return *s_ok != 0;
}

// Groups g = blockIdx.x, + gridDim.x, ...: tile offsets and counts[g].
__device__ __forceinline__ void partition_scan(const PartitionWs &w, int n_tiles, int ng,
                                               int32_t *counts, int *warp_sums, int *s_total) {
    for (int g = blockIdx.x; g < ng; g += gridDim.x) {
        int carry = 0;
        for (int base = 0; base < n_tiles; base += blockDim.x) {
            const int tile = base + static_cast<int>(threadIdx.x);
            int c = 0;
            if (tile < n_tiles) {
                const uint4 b =
                    __ldcg(reinterpret_cast<const uint4 *>(w.bal + (static_cast<size_t>(tile) * ng + g) * 4));
                c = __popc(b.x) + __popc(b.y) + __popc(b.z) + __popc(b.w);
            }
            const int ex = block_exclusive_scan(c, warp_sums, s_total);
            if (tile < n_tiles) w.off[static_cast<size_t>(tile) * ng + g] = carry + ex;
            carry += *s_total;
            __syncthreads();
        }
        if (threadIdx.x == 0) counts[g] = carry;
    }
}

// Tiles tile = blockIdx.x, + gridDim.x, ...: every token's place in perm[g].
// scratch: at least 24 * ng bytes of shared memory, 16-byte aligned.
__device__ __forceinline__ void partition_place(const PartitionWs &w, int n_tiles, int ng, int T,
                                                const int32_t *counts, int32_t *perm, uint8_t *scratch) {
    uint32_t *sb = reinterpret_cast<uint32_t *>(scratch);  // [ng][4] ballots
    int *so = reinterpret_cast<int *>(sb + ng * 4);        // [ng] tile offsets
    int *sc = so + ng;                                     // [ng] counts
    for (int i = threadIdx.x; i < ng; i += blockDim.x) sc[i] = __ldcg(counts + i);
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        for (int i = threadIdx.x; i < ng; i += blockDim.x) {
            reinterpret_cast<uint4 *>(sb)[i] =
                __ldcg(reinterpret_cast<const uint4 *>(w.bal + (static_cast<size_t>(tile) * ng + i) * 4));
            so[i] = __ldcg(w.off + static_cast<size_t>(tile) * ng + i);
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < ng * kPartTile; idx += blockDim.x) {
            const int g = idx / kPartTile, r = idx - g * kPartTile;
            const int t = tile * kPartTile + r;
            if (t >= T) continue;
            const uint4 b = reinterpret_cast<const uint4 *>(sb)[g];
            const int q = r >> 5, ln = r & 31;
            const uint32_t wq = q == 0 ? b.x : q == 1 ? b.y : q == 2 ? b.z : b.w;
            int before = __popc(wq & ((1u << ln) - 1u));
            if (q > 0) before += __popc(b.x);
            if (q > 1) before += __popc(b.y);
            if (q > 2) before += __popc(b.z);
            const int a_off = so[g];
            const int pos = ((wq >> ln) & 1u) ? a_off + before : sc[g] + (tile * kPartTile - a_off) + (r - before);
            perm[static_cast<size_t>(g) * T + pos] = t;
        }
        __syncthreads();
    }
}

}  // namespace wide
