// loss.cu -- fused GRPO / PPO clipped-ratio loss fragment.
//
// "RL-Kernel integration roadmap for vime", RL Loss Operators: fused
// ratio / loss fragments whose contract fixes mask handling, aggregation,
// dtype and reduction order, while the caller owns the algorithm (advantages,
// clipping range, aggregation).  "RL-Kernel Roadmap (2026)", backlog: fused
// PPO clip loss, generalized ratio-clip-aggregate policy-gradient primitive.
//
// For active t, r_t = exp(logp_t - old_t) (fp32, expf), lo = 1 - eps_low,
// hi = 1 + eps_high:
//   term_t = min(r_t A_t, clip(r_t, lo, hi) A_t)
//   g_t    = (-A_t r_t) * scale   when the unclipped product is the min, else 0
//   loss   = -scale * sum_active term_t
// plus the active count, the zero-gradient clipped count, the out-of-range
// count and the mean ratio.  g_t depends on token t alone (and on the
// caller's scale), so it is batch invariant.  Reductions: fixed 4096-element
// blocks, fp32 per-thread sums in ascending index order, fp64 fixed shuffle
// trees, and a single-block merge launched with programmatic dependent launch.
#include <cmath>

#include "rlk_internal.h"

namespace rlk {

namespace {

struct LossAcc {
    int64_t count, clipped, outside;
    double sum_term, sum_r;
};

__device__ __forceinline__ void add(LossAcc& a, const LossAcc& b) {
    a.count += b.count;
    a.clipped += b.clipped;
    a.outside += b.outside;
    a.sum_term += b.sum_term;
    a.sum_r += b.sum_r;
}

__device__ __forceinline__ LossAcc shfl_down(const LossAcc& a, int off) {
    LossAcc b;
    b.count = __shfl_down_sync(0xffffffffu, a.count, off);
    b.clipped = __shfl_down_sync(0xffffffffu, a.clipped, off);
    b.outside = __shfl_down_sync(0xffffffffu, a.outside, off);
    b.sum_term = __shfl_down_sync(0xffffffffu, a.sum_term, off);
    b.sum_r = __shfl_down_sync(0xffffffffu, a.sum_r, off);
    return b;
}

template <int THREADS>
__device__ __forceinline__ LossAcc block_sum(LossAcc a) {
    __shared__ LossAcc warp_acc[THREADS / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        LossAcc b = shfl_down(a, off);
        if (lane + off < 32) add(a, b);
    }
    if (lane == 0) warp_acc[warp] = a;
    __syncthreads();
    if (warp == 0) {
        a = lane < THREADS / 32 ? warp_acc[lane] : LossAcc{0, 0, 0, 0.0, 0.0};
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            LossAcc b = shfl_down(a, off);
            if (lane + off < 32) add(a, b);
        }
    }
    return a;
}

struct ThreadSums {
    int count = 0, clipped = 0, outside = 0;     // at most kLossPerThread each
    float term = 0.f, r = 0.f;
};

__device__ __forceinline__ float token(float nw, float od, float adv, uint8_t m, float lo, float hi,
                                       float scale, ThreadSums& s) {
    if (m == 0) return 0.f;
    const float r = expf(nw - od);
    const float rc = fminf(fmaxf(r, lo), hi);
    const float u = r * adv;
    const float c = rc * adv;
    const bool take = u <= c;
    const bool out = (r < lo) || (r > hi);
    ++s.count;
    s.clipped += (!take && out) ? 1 : 0;
    s.outside += out ? 1 : 0;
    s.term += take ? u : c;
    s.r += r;
    return take ? (-adv * r) * scale : 0.f;
}

template <bool VEC>
__global__ void __launch_bounds__(kAuditThreads)
    loss_pass1(const float* __restrict__ nw, const float* __restrict__ od,
               const float* __restrict__ adv, const uint8_t* __restrict__ mask, int64_t N,
               float lo, float hi, float scale, float* __restrict__ grad,
               LossPartial* __restrict__ out) {
    asm volatile("griddepcontrol.launch_dependents;");
    constexpr int kVec = kLossPerThread / 4;
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kLossBlockElems;
    ThreadSums s;
    if (VEC && base + kLossBlockElems <= N) {
        float4 a[kVec], b[kVec], c[kVec];
        uint32_t m[kVec];
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const int64_t i0 = base + j * (kAuditThreads * 4) + threadIdx.x * 4;
            a[j] = __ldcs(reinterpret_cast<const float4*>(nw + i0));
            b[j] = __ldcs(reinterpret_cast<const float4*>(od + i0));
            c[j] = __ldcs(reinterpret_cast<const float4*>(adv + i0));
            m[j] = mask == nullptr ? 0x01010101u
                                   : __ldcs(reinterpret_cast<const unsigned int*>(mask + i0));
        }
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const int64_t i0 = base + j * (kAuditThreads * 4) + threadIdx.x * 4;
            float4 g;
            g.x = token(a[j].x, b[j].x, c[j].x, uint8_t(m[j]), lo, hi, scale, s);
            g.y = token(a[j].y, b[j].y, c[j].y, uint8_t(m[j] >> 8), lo, hi, scale, s);
            g.z = token(a[j].z, b[j].z, c[j].z, uint8_t(m[j] >> 16), lo, hi, scale, s);
            g.w = token(a[j].w, b[j].w, c[j].w, uint8_t(m[j] >> 24), lo, hi, scale, s);
            __stcs(reinterpret_cast<float4*>(grad + i0), g);
        }
    } else {
#pragma unroll 1
        for (int j = 0; j < kVec; ++j) {
            const int64_t i0 = base + j * (kAuditThreads * 4) + threadIdx.x * 4;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int64_t i = i0 + e;
                if (i < N)
                    grad[i] = token(nw[i], od[i], adv[i], mask == nullptr ? uint8_t(1) : mask[i],
                                    lo, hi, scale, s);
            }
        }
    }
    LossAcc acc{s.count, s.clipped, s.outside, static_cast<double>(s.term),
                static_cast<double>(s.r)};
    acc = block_sum<kAuditThreads>(acc);
    if (threadIdx.x == 0) {
        LossPartial p;
        p.count = acc.count;
        p.clipped = acc.clipped;
        p.outside = acc.outside;
        p.sum_term = acc.sum_term;
        p.sum_r = acc.sum_r;
        out[blockIdx.x] = p;
    }
}

constexpr int kLossMergeThreads = 1024;

__global__ void __launch_bounds__(kLossMergeThreads)
    loss_pass2(const LossPartial* __restrict__ parts, int64_t num_parts, double scale,
               rlk_grpo_result_t* __restrict__ result) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    LossAcc a{0, 0, 0, 0.0, 0.0};
    // thread t adds partials t, t + T, t + 2T, ... in ascending order, loading four at a
    // time so that the loads overlap (the order of the additions is unchanged)
    int64_t i = threadIdx.x;
    for (; i + 3 * kLossMergeThreads < num_parts; i += 4 * kLossMergeThreads) {
        LossPartial p[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) p[j] = parts[i + j * kLossMergeThreads];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            add(a, LossAcc{p[j].count, p[j].clipped, p[j].outside, p[j].sum_term, p[j].sum_r});
    }
    for (; i < num_parts; i += kLossMergeThreads) {
        const LossPartial p = parts[i];
        add(a, LossAcc{p.count, p.clipped, p.outside, p.sum_term, p.sum_r});
    }
    a = block_sum<kLossMergeThreads>(a);
    if (threadIdx.x == 0) {
        rlk_grpo_result_t r;
        r.active_count = a.count;
        r.clipped_count = a.clipped;
        r.outside_count = a.outside;
        r.loss = -scale * a.sum_term;
        r.mean_ratio = a.sum_r / static_cast<double>(a.count);
        *result = r;
    }
}

}  // namespace

cudaError_t launch_grpo_loss(const float* logp_new, const float* logp_old, const float* adv,
                             const uint8_t* mask, int64_t N, double eps_low, double eps_high,
                             double scale, float* grad, rlk_grpo_result_t* result,
                             void* workspace, bool vec_ok, cudaStream_t stream) {
    const size_t blocks = loss_blocks(N);
    LossPartial* parts = static_cast<LossPartial*>(workspace);
    const float lo = static_cast<float>(1.0 - eps_low);
    const float hi = static_cast<float>(1.0 + eps_high);
    const float sc = static_cast<float>(scale);
    if (blocks > 0) {
        if (vec_ok)
            loss_pass1<true><<<static_cast<unsigned>(blocks), kAuditThreads, 0, stream>>>(
                logp_new, logp_old, adv, mask, N, lo, hi, sc, grad, parts);
        else
            loss_pass1<false><<<static_cast<unsigned>(blocks), kAuditThreads, 0, stream>>>(
                logp_new, logp_old, adv, mask, N, lo, hi, sc, grad, parts);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kLossMergeThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const LossPartial* cparts = parts;
    const int64_t nparts = static_cast<int64_t>(blocks);
    return cudaLaunchKernelEx(&cfg, loss_pass2, cparts, nparts, scale, result);
}

}  // namespace rlk
