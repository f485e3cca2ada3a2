// compact.cu -- active-row compaction for masked batches.
//
// "RL-Kernel integration roadmap for vime", Consistency Contract: all metrics
// use active tokens only, and a token's result must not change with padding,
// packing or active-mask density.  The forward GEMM therefore only needs the
// active rows: they are gathered, in ascending token order, into a contiguous
// buffer, so padding and masked-out tokens cost no tensor-core work.  A row's
// arithmetic does not depend on the tile it lands in, so the result is bitwise
// the same as without compaction.
//
// Deterministic and atomic-free: kernel 1 counts the active rows of each
// 1024-row block; kernel 2 gives each block its offset as the sum of the counts
// before it (summed by all the block's threads), places the block's active rows by warp
// ballots (ascending token order), records rows[pos] = t and pos_of[t] = pos
// (-1 for inactive rows), and block 0 stores the active count; kernel 3 copies
// the active rows of h, one warp per row over a grid that covers every row, and
// zeroes the rows after them up to the end of the last 128-row block (at least
// one block), so the backward's K loop over the compacted rows (64-row K blocks)
// never meets stale bytes.  GEMM rows past the active count are dead rows: the
// epilogues discard them, or write zeros whatever their accumulators hold.
//
// In the backward the inactive tokens are never visited by a GEMM, so their
// rows of dh are zeroed by a fourth kernel.
#include "rlk_internal.h"

namespace rlk {

namespace {

constexpr int kCompactThreads = kCompactBlock;

__global__ void __launch_bounds__(kCompactThreads)
    compact_count_kernel(const uint8_t* __restrict__ mask, int N, int* __restrict__ blk_count) {
    const int t = blockIdx.x * kCompactThreads + threadIdx.x;
    const bool act = t < N && mask[t] != 0;
    const unsigned ballot = __ballot_sync(0xffffffffu, act);
    __shared__ int warp_count[kCompactThreads / 32];
    if ((threadIdx.x & 31) == 0) warp_count[threadIdx.x >> 5] = __popc(ballot);
    __syncthreads();
    if (threadIdx.x == 0) {
        int c = 0;
        for (int w = 0; w < kCompactThreads / 32; ++w) c += warp_count[w];
        blk_count[blockIdx.x] = c;
    }
}

__global__ void __launch_bounds__(kCompactThreads)
    compact_place_kernel(const uint8_t* __restrict__ mask, int N,
                         const int* __restrict__ blk_count, int num_blocks,
                         int* __restrict__ rows, int* __restrict__ pos_of,
                         int* __restrict__ n_active) {
    __shared__ int s_base;
    __shared__ int warp_count[kCompactThreads / 32];
    __shared__ int warp_off[kCompactThreads / 32];
    __shared__ int s_part[kCompactThreads / 32];
    // this block's offset: the counts of the blocks before it, summed by all threads
    // (integers: the order of the additions does not matter); block 0 also sums them all
    {
        const int upto = blockIdx.x == 0 ? num_blocks : static_cast<int>(blockIdx.x);
        int part = 0;
        for (int b = threadIdx.x; b < upto; b += kCompactThreads) part += blk_count[b];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_down_sync(0xffffffffu, part, off);
        if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = part;
        __syncthreads();
        if (threadIdx.x == 0) {
            int sum = 0;
            for (int w = 0; w < kCompactThreads / 32; ++w) sum += s_part[w];
            s_base = blockIdx.x == 0 ? 0 : sum;
            if (blockIdx.x == 0) *n_active = sum;
        }
    }
    const int t = blockIdx.x * kCompactThreads + threadIdx.x;
    const bool act = t < N && mask[t] != 0;
    const unsigned ballot = __ballot_sync(0xffffffffu, act);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) warp_count[warp] = __popc(ballot);
    __syncthreads();
    if (threadIdx.x == 0) {
        int off = 0;
        for (int w = 0; w < kCompactThreads / 32; ++w) {
            warp_off[w] = off;
            off += warp_count[w];
        }
    }
    __syncthreads();
    const int pos = s_base + warp_off[warp] + __popc(ballot & ((1u << lane) - 1u));
    if (t < N) {
        pos_of[t] = act ? pos : -1;
        if (act) rows[pos] = t;
    }
}

constexpr int kGatherWarps = 8;             // rows per block of the copy

// hidden_c[i] = hidden[rows[i]] for i < n_active, zero for the rows after them
// up to the end of their last tile: one warp per row, 16 bytes per lane and access
__global__ void __launch_bounds__(kGatherWarps * 32)
    compact_gather_kernel(const int* __restrict__ rows, const int* __restrict__ n_active, int N,
                          int H, const uint4* __restrict__ hidden, uint4* __restrict__ hidden_c) {
    const int i = blockIdx.x * kGatherWarps + (threadIdx.x >> 5);
    const int n = *n_active;
    const int pad_end = min(N, (max(n, 1) + kTileM - 1) / kTileM * kTileM);
    if (i >= pad_end) return;
    const int lane = threadIdx.x & 31;
    const int vec_per_row = H / 8;
    uint4* dst = hidden_c + static_cast<size_t>(i) * vec_per_row;
    if (i < n) {
        const uint4* src = hidden + static_cast<size_t>(rows[i]) * vec_per_row;
        for (int j = lane; j < vec_per_row; j += 32) dst[j] = src[j];
    } else {
        for (int j = lane; j < vec_per_row; j += 32) dst[j] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// out[t] = 0 for every inactive token t: one warp per row, 16-byte stores
__global__ void __launch_bounds__(kGatherWarps * 32)
    zero_inactive_rows_kernel(const uint8_t* __restrict__ mask, int N, int vec_per_row,
                              uint4* __restrict__ out) {
    const int t = blockIdx.x * kGatherWarps + (threadIdx.x >> 5);
    if (t >= N || mask[t] != 0) return;
    uint4* dst = out + static_cast<size_t>(t) * vec_per_row;
    for (int j = threadIdx.x & 31; j < vec_per_row; j += 32) dst[j] = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace

cudaError_t launch_compact(const uint8_t* mask, int N, int H, const void* hidden, void* hidden_c,
                           int* blk_count, int* rows, int* pos_of, int* n_active,
                           cudaStream_t stream) {
    const int blocks = (N + kCompactThreads - 1) / kCompactThreads;
    compact_count_kernel<<<blocks, kCompactThreads, 0, stream>>>(mask, N, blk_count);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    compact_place_kernel<<<blocks, kCompactThreads, 0, stream>>>(mask, N, blk_count, blocks, rows,
                                                                 pos_of, n_active);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    compact_gather_kernel<<<(N + kGatherWarps - 1) / kGatherWarps, kGatherWarps * 32, 0, stream>>>(
        rows, n_active, N, H, static_cast<const uint4*>(hidden), static_cast<uint4*>(hidden_c));
    return cudaGetLastError();
}

cudaError_t launch_zero_inactive_rows(const uint8_t* mask, int N, size_t row_bytes, void* out,
                                      cudaStream_t stream) {
    zero_inactive_rows_kernel<<<(N + kGatherWarps - 1) / kGatherWarps, kGatherWarps * 32, 0,
                                stream>>>(mask, N, static_cast<int>(row_bytes / 16),
                                          static_cast<uint4*>(out));
    return cudaGetLastError();
}

}  // namespace rlk
