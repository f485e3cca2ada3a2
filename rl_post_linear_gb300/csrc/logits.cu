// logits.cu -- selected-token logp from existing logits.
//
// "RL-Kernel integration roadmap for vime", logp Reference Scoring: the
// audit / reference sibling of linear_logp for when logits already exist, with
// an explicit log-softmax contract (max and sum-exp dtype and order, downcast
// point) and a deterministic row-local policy: fixed reduction topology,
// fixed launch configuration, bitwise equal results for dense and indexed rows
// and whatever the batch.
//
// One CTA of 256 threads scores one row.  Thread j owns the column groups
// g = j, j + 256, j + 512, ... (a group is 4 fp32 or 8 bf16 consecutive
// columns) and folds them in ascending order into an fp32 running
// (max m, sum s = sum 2^((x - m) k)), k = log2(e)/T; the 256 pairs are then
// merged by a fixed shuffle tree.  None of this depends on N, on the row's
// position or on whether the row was picked by an index list.
#include <cuda_bf16.h>

#include <cmath>

#include "ptx.cuh"
#include "rlk_internal.h"

namespace rlk {

namespace {

constexpr int kLogitsThreads = 256;

struct MS {
    float m, s;
};

__device__ __forceinline__ MS combine(MS a, MS b, float k) {
    if (b.m == -INFINITY) return a;
    if (a.m == -INFINITY) return b;
    const float m = fmaxf(a.m, b.m);
    return MS{m, a.s * ex2_approx((a.m - m) * k) + b.s * ex2_approx((b.m - m) * k)};
}

template <int VEC>
__device__ __forceinline__ void fold(float (&x)[VEC], int valid, float k, MS& st) {
    float gm = -INFINITY;
#pragma unroll
    for (int e = 0; e < VEC; ++e)
        if (e < valid) gm = fmaxf(gm, x[e]);
    if (gm > st.m) {
        st.s = st.s * ex2_approx((st.m - gm) * k);
        st.m = gm;
    }
#pragma unroll
    for (int e = 0; e < VEC; ++e)
        if (e < valid) st.s += ex2_approx((x[e] - st.m) * k);
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__global__ void __launch_bounds__(kLogitsThreads)
    logp_from_logits_kernel(const T* __restrict__ logits, int64_t stride, int64_t N, int V,
                            const int64_t* __restrict__ rows, const int64_t* __restrict__ targets,
                            const uint8_t* __restrict__ mask, float k, bool vec_ok,
                            float* __restrict__ logp, float* __restrict__ lse, uint32_t* err) {
    constexpr int VEC = 16 / sizeof(T);
    const int i = blockIdx.x;
    const int64_t r = rows != nullptr ? rows[i] : i;
    if (r < 0 || r >= N) {                  // an index list entry outside the logits
        if (threadIdx.x == 0) {
            logp[i] = __int_as_float(0x7fc00000);
            if (lse != nullptr) lse[i] = __int_as_float(0x7fc00000);
            if (err != nullptr) atomicOr(err, RLK_DEVERR_ROW_RANGE);
        }
        return;
    }
    if (mask != nullptr && mask[r] == 0) {
        if (threadIdx.x == 0) {
            logp[i] = 0.f;
            if (lse != nullptr) lse[i] = 0.f;
        }
        return;
    }
    const T* row = logits + r * stride;
    MS st{-INFINITY, 0.f};
    const int groups = (V + VEC - 1) / VEC;
    int g = threadIdx.x;
    if (vec_ok) {
        // four of the thread's groups per step, all loads first (more bytes in flight);
        // they are folded in the same ascending order as one at a time
        const int full = V / VEC;                // groups with VEC valid columns
        for (; g + 3 * kLogitsThreads < full; g += 4 * kLogitsThreads) {
            uint4 raw[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                raw[q] = __ldcs(reinterpret_cast<const uint4*>(row + (g + q * kLogitsThreads) * VEC));
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const T* v = reinterpret_cast<const T*>(&raw[q]);
                float x[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) x[e] = to_f32(v[e]);
                fold<VEC>(x, VEC, k, st);
            }
        }
    }
    for (; g < groups; g += kLogitsThreads) {
        const int c0 = g * VEC;
        const int valid = min(VEC, V - c0);
        float x[VEC];
        if (vec_ok && valid == VEC) {
            const uint4 raw = __ldcs(reinterpret_cast<const uint4*>(row + c0));
            const T* v = reinterpret_cast<const T*>(&raw);
#pragma unroll
            for (int e = 0; e < VEC; ++e) x[e] = to_f32(v[e]);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) x[e] = e < valid ? to_f32(row[c0 + e]) : -INFINITY;
        }
        fold<VEC>(x, valid, k, st);
    }
    // fixed tree: lanes, then warps in order
    __shared__ MS warp_ms[kLogitsThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        MS o{__shfl_down_sync(0xffffffffu, st.m, off), __shfl_down_sync(0xffffffffu, st.s, off)};
        if (lane + off < 32) st = combine(st, o, k);
    }
    if (lane == 0) warp_ms[warp] = st;
    __syncthreads();
    if (warp != 0) return;
    st = lane < kLogitsThreads / 32 ? warp_ms[lane] : MS{-INFINITY, 0.f};
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        MS o{__shfl_down_sync(0xffffffffu, st.m, off), __shfl_down_sync(0xffffffffu, st.s, off)};
        if (lane + off < 32) st = combine(st, o, k);
    }
    if (lane != 0) return;
    constexpr float kLn2 = 0.693147180559945309f;
    const float lse2 = st.m * k + lg2_approx(st.s);
    if (lse != nullptr) lse[i] = lse2 * kLn2;
    const int64_t y = targets[r];
    if (y < 0 || y >= V) {
        logp[i] = __int_as_float(0x7fc00000);
        if (err != nullptr) atomicOr(err, RLK_DEVERR_TARGET_RANGE);
        return;
    }
    logp[i] = (to_f32(row[y]) * k - lse2) * kLn2;
}

}  // namespace

cudaError_t launch_logp_from_logits(const void* logits, bool bf16, int64_t stride, int64_t N, int V,
                                    const int64_t* rows, int M, const int64_t* targets,
                                    const uint8_t* mask, float k, bool vec_ok, float* logp,
                                    float* lse, uint32_t* err, cudaStream_t stream) {
    if (M == 0) return cudaSuccess;
    if (bf16)
        logp_from_logits_kernel<__nv_bfloat16><<<M, kLogitsThreads, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(logits), stride, N, V, rows, targets, mask, k, vec_ok,
            logp, lse, err);
    else
        logp_from_logits_kernel<float><<<M, kLogitsThreads, 0, stream>>>(
            static_cast<const float*>(logits), stride, N, V, rows, targets, mask, k, vec_ok, logp,
            lse, err);
    return cudaGetLastError();
}

}  // namespace rlk
