// reorder.cu -- mask reordering (WIDE, Sec. 3.3 Eq. 7; App. B Algorithm 1).
//
// One CTA per routing column g (the columns are independent, as Algorithm 1
// states).  Each thread owns a run of up to 32 consecutive tokens, packs their
// mask bits into one register, and a block-wide exclusive scan of the per-run
// active counts gives every run its output positions: active tokens go to
// the prefix in ascending order, inactive tokens after counts[g] in
// ascending order.  Columns longer than 32 * blockDim tokens are processed in
// chunks after a counting pass.
#include "common.cuh"
#include "internal.h"

namespace wide {
namespace {

constexpr int kThreads = 1024;
constexpr int kRun = 32;  // tokens per thread per chunk (one bit each)

// Exclusive scan of v over the block; *total receives the block sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_sums, int *total) {
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
    const int g = blockIdx.x;
    const int tid = threadIdx.x;
    const long long chunk = static_cast<long long>(kThreads) * kRun;
    int32_t *out = perm + static_cast<size_t>(g) * T;

    int total = -1;  // active rows in the whole column, once known
    if (T > chunk) {
        int c = 0;
        for (long long t = tid; t < T; t += kThreads)
            c += mask[static_cast<size_t>(t) * n_groups + g] != 0;
        block_exclusive_scan(c, warp_sums, &s_total);
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
#pragma unroll 8
        for (int j = 0; j < kRun; ++j) {
            if (j < n_tok) {
                const size_t t = static_cast<size_t>(base + first + j);
                bits |= static_cast<uint32_t>(mask[t * n_groups + g] != 0) << j;
            }
        }
        const int n_act = __popc(bits);
        const int a_off = block_exclusive_scan(n_act, warp_sums, &s_total);
        __syncthreads();
        const int chunk_active = s_total;
        if (total < 0) total = chunk_active;  // single chunk: column total known now
        const int tok_before = min(first, len);
        int pa = run_active + a_off;
        int pi = total + static_cast<int>(base - run_active) + (tok_before - a_off);
        for (int j = 0; j < n_tok; ++j) {
            const int t = static_cast<int>(base) + first + j;
            if ((bits >> j) & 1u) out[pa++] = t;
            else out[pi++] = t;
        }
        run_active += chunk_active;
        __syncthreads();
    }
    if (tid == 0) counts[g] = total;
}

}  // namespace

cudaError_t launch_reorder(const uint8_t *mask, int T, int n_groups, int32_t *perm,
                           int32_t *counts, cudaStream_t s) {
    reorder_kernel<<<n_groups, kThreads, 0, s>>>(mask, T, n_groups, perm, counts);
    return cudaGetLastError();
}

}  // namespace wide
