// reorder.cu -- mask reordering (WIDE, Sec. 3.3 Eq. 7; App. B Algorithm 1).
//
// One CTA per routing column g (the columns are independent, as Algorithm 1
// states).  Each thread owns a run of up to 32 consecutive tokens, packs their
// mask bits into one register, and a block-wide exclusive scan of the per-run
// active counts gives every run its output positions: active tokens go to
// the prefix in ascending order, inactive tokens after counts[g] in
// ascending order.  Columns longer than 32 * blockDim tokens are processed in
// chunks after a counting pass.  Each chunk's partition is assembled in shared
// memory and copied out as two contiguous ranges (coalesced stores).  This
// kernel reads each column at a stride of n_groups bytes.
//
// With a workspace, reorder_coop_kernel does the same partition from
// coalesced reads of the mask rows instead: a cooperative grid stages each
// 128-token tile's mask rows in shared memory, ballots every group over the
// tile's four 32-token warps, and finishes with the scan and placement of
// partition.cuh (grid barriers between the phases).
#include "common.cuh"
#include "internal.h"
#include "partition.cuh"

namespace wide {
namespace {

constexpr int kThreads = 1024;
constexpr int kRun = 32;  // tokens per thread per chunk (one bit each)
constexpr int kCoopThreads = 256;
constexpr int kGroupChunk = 128;  // mask columns staged per pass

// Exclusive scan of v over the block; *total receives the block sum.
__device__ __forceinline__ int column_exclusive_scan(int v, int *warp_sums, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += y;
    }
    if (lane == 31) warp_sums[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        int w = lane < nw ? warp_sums[lane] : 0;
        int winc = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, winc, d);
            if (lane >= d) winc += y;
        }
        warp_sums[lane] = winc - w;  // exclusive prefix of warp totals
        if (lane == 31) *total = winc;
    }
    __syncthreads();
    const int out = warp_sums[warp] + inc - v;
    __syncthreads();  // warp_sums may be reused by the caller's next scan
    return out;
}

__global__ void __launch_bounds__(kThreads)
    reorder_kernel(const uint8_t *__restrict__ mask, int T, int n_groups,
                   int32_t *__restrict__ perm, int32_t *__restrict__ counts) {
    __shared__ int warp_sums[32];
    __shared__ int s_total;
    // this chunk's partition (its active tokens, then its inactive ones), copied
    // out as two contiguous ranges so that the stores coalesce
    extern __shared__ int32_t s_part[];
    const int g = blockIdx.x;
    const int tid = threadIdx.x;
    const long long chunk = static_cast<long long>(kThreads) * kRun;
    int32_t *out = perm + static_cast<size_t>(g) * T;

    int total = -1;  // active rows in the whole column, once known
    if (T > chunk) {
        int c = 0;
        for (long long t = tid; t < T; t += kThreads)
            c += mask[static_cast<size_t>(t) * n_groups + g] != 0;
        column_exclusive_scan(c, warp_sums, &s_total);
        __syncthreads();
        total = s_total;
    }

    int run_active = 0;  // active rows before the current chunk
    for (long long base = 0; base < T; base += chunk) {
        const long long rem = static_cast<long long>(T) - base;
        const int len = static_cast<int>(rem < chunk ? rem : chunk);
        const int R = (len + kThreads - 1) / kThreads;  // <= kRun
        const int first = tid * R;                      // offset inside the chunk
        const int n_tok = max(0, min(R, len - first));
        uint32_t bits = 0;
#pragma unroll
        for (int j = 0; j < kRun; ++j) {
            if (j < n_tok) {
                const size_t t = static_cast<size_t>(base + first + j);
                bits |= static_cast<uint32_t>(mask[t * n_groups + g] != 0) << j;
            }
        }
        const int n_act = __popc(bits);
        const int a_off = column_exclusive_scan(n_act, warp_sums, &s_total);
        __syncthreads();
        const int chunk_active = s_total;
        if (total < 0) total = chunk_active;  // single chunk: column total known now
        const int tok_before = min(first, len);
        int la = a_off;                                  // chunk-local slots
        int li = chunk_active + (tok_before - a_off);
        for (int j = 0; j < n_tok; ++j) {
            const int t = static_cast<int>(base) + first + j;
            if ((bits >> j) & 1u) s_part[la++] = t;
            else s_part[li++] = t;
        }
        __syncthreads();
        // active tokens go to run_active.., inactive ones to total + (inactive before)..
        const long long ina_dst = total + (base - run_active) - chunk_active;
        for (int i = tid; i < len; i += kThreads)
            out[i < chunk_active ? run_active + i : static_cast<int>(ina_dst + i)] = s_part[i];
        run_active += chunk_active;
        __syncthreads();
    }
    if (tid == 0) counts[g] = total;
}

// Cooperative stable partition: ballots of each tile (coalesced row reads
// staged in shared memory), then partition_scan / partition_place.
__global__ void __launch_bounds__(kCoopThreads)
    reorder_coop_kernel(const uint8_t *__restrict__ mask, int T, int ng, int32_t *__restrict__ perm,
                        int32_t *__restrict__ counts, uint32_t *ws, int *status) {
    extern __shared__ __align__(16) uint8_t smem[];  // [128][kGroupChunk] mask bytes, then scratch
    __shared__ int warp_sums[32];
    __shared__ int s_total;
    __shared__ int s_ok;
    const int n_tiles = (T + kPartTile - 1) / kPartTile;
    const PartitionWs w = partition_ws(ws, n_tiles, ng);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;  // this warp's 32-token quarter of the tile
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int t0 = tile * kPartTile;
        for (int g0 = 0; g0 < ng; g0 += kGroupChunk) {
            const int gc = min(kGroupChunk, ng - g0);
            for (int i = threadIdx.x; i < kPartTile * gc; i += kCoopThreads) {
                const int r = i / gc, c = i - r * gc;
                const int t = t0 + r;
                smem[r * kGroupChunk + c] = t < T ? mask[static_cast<size_t>(t) * ng + g0 + c] : 0;
            }
            __syncthreads();
            // warps 0-3 and 4-7 take alternate groups; each ballots its quarter
            for (int c = warp >> 2; c < gc; c += kCoopThreads / 128) {
                const uint32_t b = __ballot_sync(0xffffffffu, smem[(q * 32 + lane) * kGroupChunk + c] != 0);
                if (lane == 0) w.bal[(static_cast<size_t>(tile) * ng + g0 + c) * 4 + q] = b;
            }
            __syncthreads();
        }
    }
    const bool ok1 = grid_barrier(w.ctr, gridDim.x, status, &s_ok);
    if (ok1) partition_scan(w, n_tiles, ng, counts, warp_sums, &s_total);
    const bool ok2 = grid_barrier(w.ctr, 2u * gridDim.x, status, &s_ok);
    if (!ok1 || !ok2) return;
    partition_place(w, n_tiles, ng, T, counts, perm, smem + kPartTile * kGroupChunk);
}

}  // namespace

size_t reorder_coop_smem_bytes(int n_groups) {
    return static_cast<size_t>(kPartTile) * kGroupChunk + static_cast<size_t>(n_groups) * 24;
}

cudaError_t launch_reorder_coop(const uint8_t *mask, int T, int n_groups, int32_t *perm, int32_t *counts,
                                uint32_t *ws, int *status, int num_sms, cudaStream_t s) {
    const size_t smem = reorder_coop_smem_bytes(n_groups);
    cudaError_t e = cudaFuncSetAttribute(reorder_coop_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reorder_coop_kernel, kCoopThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    const int tiles = (T + kPartTile - 1) / kPartTile;
    const int grid = tiles < per_sm * num_sms ? tiles : per_sm * num_sms;  // every CTA resident
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kCoopThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, reorder_coop_kernel, mask, T, n_groups, perm, counts, ws, status);
}

cudaError_t launch_reorder(const uint8_t *mask, int T, int n_groups, int32_t *perm,
                           int32_t *counts, cudaStream_t s) {
    const long long chunk = static_cast<long long>(kThreads) * kRun;
    const int smem = static_cast<int>((T < chunk ? T : chunk) * sizeof(int32_t));
    cudaError_t e = cudaFuncSetAttribute(reorder_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(chunk * sizeof(int32_t)));
    if (e != cudaSuccess) return e;
    reorder_kernel<<<n_groups, kThreads, smem, s>>>(mask, T, n_groups, perm, counts);
    return cudaGetLastError();
}

}  // namespace wide
