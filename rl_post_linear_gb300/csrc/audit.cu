// audit.cu -- deterministic masked dlogp audit.
//
// "RL-Kernel integration roadmap for vime", Consistency Contract:
// dlogp = recomputed - old; every aggregate over active tokens only;
// max_abs_dlogp is the primary metric, reported with the worst token;
// approx_kl0 = mean(exp(dlogp) - 1 - dlogp); the active-token count.
//
// Pass 1: block b owns the fixed slice [b*4096, (b+1)*4096) (a function of N
// only).  Each thread handles 16 elements in ascending index order:
// d = new - old in fp32 (a correctly rounded difference), its count, the
// largest |d| with the first index attaining it, and fp32 sums of d and of
// kl(d) = exp(d) - 1 - d.  The sums go to fp64 for a fixed shuffle tree
// (lanes, then warps).  Pass 2: one block merges the per-block partials,
// each thread a fixed strided subset in ascending order, then the same
// fixed tree.  No atomics; the result is bitwise reproducible for a given N.
//
// kl(d) for |d| < 1/2 is the Taylor series d^2 (1/2 + d/6 + d^2/24 + ...)
// through the d^9 term (truncation below 3e-9 relative); elsewhere it is
// expm1f(d) - d, where no cancellation arises.
#include <cmath>
#include <mutex>

#include "rlk_internal.h"

namespace rlk {

namespace {

__device__ __forceinline__ float kl_term(float d) {
    if (fabsf(d) < 0.5f) {
        float p = 1.0f / 362880.0f;
        p = fmaf(p, d, 1.0f / 40320.0f);
        p = fmaf(p, d, 1.0f / 5040.0f);
        p = fmaf(p, d, 1.0f / 720.0f);
        p = fmaf(p, d, 1.0f / 120.0f);
        p = fmaf(p, d, 1.0f / 24.0f);
        p = fmaf(p, d, 1.0f / 6.0f);
        p = fmaf(p, d, 0.5f);
        return d * d * p;
    }
    return expm1f(d) - d;
}

// (a1, i1) ranks strictly above (a2, i2): NaN above every number, then the
// larger |d|, then the lower index.
__device__ __forceinline__ bool ranks_above(float a1, int64_t i1, float a2, int64_t i2) {
    const bool n1 = isnan(a1), n2 = isnan(a2);
    if (n1 != n2) return n1;
    if (!n1 && a1 != a2) return a1 > a2;
    return i1 < i2;
}

struct Acc {
    int64_t count;
    int64_t arg;
    double sum_d;
    double sum_kl;
    float best;
    uint32_t flags;
};

__device__ __forceinline__ Acc empty_acc() {
    Acc a;
    a.count = 0;
    a.arg = INT64_MAX;
    a.sum_d = 0.0;
    a.sum_kl = 0.0;
    a.best = -1.0f;
    a.flags = 0;
    return a;
}

// a := a (+) b, with a covering lower indices than b
__device__ __forceinline__ void merge(Acc& a, const Acc& b) {
    a.count += b.count;
    a.sum_d += b.sum_d;
    a.sum_kl += b.sum_kl;
    a.flags |= b.flags;
    if (b.count > 0 && (a.count == b.count || ranks_above(b.best, b.arg, a.best, a.arg))) {
        a.best = b.best;
        a.arg = b.arg;
    }
}

__device__ __forceinline__ Acc shfl_down(const Acc& a, int off) {
    Acc b;
    b.count = __shfl_down_sync(0xffffffffu, a.count, off);
    b.arg = __shfl_down_sync(0xffffffffu, a.arg, off);
    b.sum_d = __shfl_down_sync(0xffffffffu, a.sum_d, off);
    b.sum_kl = __shfl_down_sync(0xffffffffu, a.sum_kl, off);
    b.best = __shfl_down_sync(0xffffffffu, a.best, off);
    b.flags = __shfl_down_sync(0xffffffffu, a.flags, off);
    return b;
}

// Fixed tree over the block: lanes (16, 8, 4, 2, 1), then the warp results
// in warp order with the same tree.  Lane 0 of warp 0 returns the total.
template <int THREADS>
__device__ __forceinline__ Acc block_reduce(Acc a) {
    __shared__ Acc warp_acc[THREADS / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Acc b = shfl_down(a, off);
        if (lane + off < 32) merge(a, b);
    }
    if (lane == 0) warp_acc[warp] = a;
    __syncthreads();
    if (warp == 0) {
        a = lane < THREADS / 32 ? warp_acc[lane] : empty_acc();
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            Acc b = shfl_down(a, off);
            if (lane + off < 32) merge(a, b);
        }
    }
    return a;
}

__device__ __forceinline__ void visit(float nw, float od, uint8_t m, int64_t idx, int64_t& count,
                                      float& best, int64_t& arg, float& sd, float& skl,
                                      uint32_t& flags) {
    if (m == 0) return;
    const float d = nw - od;
    const float a = fabsf(d);
    if (count == 0 || ranks_above(a, idx, best, arg)) {
        best = a;
        arg = idx;
    }
    ++count;
    sd += d;
    skl += kl_term(d);
    if (!isfinite(d)) flags |= 1u;
}

template <bool VEC>
__global__ void __launch_bounds__(kAuditThreads)
    audit_pass1(const float* __restrict__ nw, const float* __restrict__ od,
                const uint8_t* __restrict__ mask, int64_t N, AuditPartial* __restrict__ out) {
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kAuditBlockElems;
    int64_t count = 0, arg = INT64_MAX;
    float best = -1.0f, sd = 0.f, skl = 0.f;
    uint32_t flags = 0;
    const bool full = base + kAuditBlockElems <= N;
#pragma unroll
    for (int j = 0; j < kAuditPerThread / 4; ++j) {
        const int64_t i0 = base + j * (kAuditThreads * 4) + threadIdx.x * 4;
        if (VEC && full) {
            const float4 a = *reinterpret_cast<const float4*>(nw + i0);
            const float4 b = *reinterpret_cast<const float4*>(od + i0);
            uchar4 m = make_uchar4(1, 1, 1, 1);
            if (mask != nullptr) m = *reinterpret_cast<const uchar4*>(mask + i0);
            visit(a.x, b.x, m.x, i0, count, best, arg, sd, skl, flags);
            visit(a.y, b.y, m.y, i0 + 1, count, best, arg, sd, skl, flags);
            visit(a.z, b.z, m.z, i0 + 2, count, best, arg, sd, skl, flags);
            visit(a.w, b.w, m.w, i0 + 3, count, best, arg, sd, skl, flags);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int64_t i = i0 + e;
                if (i < N)
                    visit(nw[i], od[i], mask == nullptr ? uint8_t(1) : mask[i], i, count, best, arg,
                          sd, skl, flags);
            }
        }
    }
    Acc a;
    a.count = count;
    a.arg = arg;
    a.sum_d = static_cast<double>(sd);
    a.sum_kl = static_cast<double>(skl);
    a.best = best;
    a.flags = flags;
    a = block_reduce<kAuditThreads>(a);
    if (threadIdx.x == 0) {
        AuditPartial p;
        p.count = a.count;
        p.arg = a.arg;
        p.sum_d = a.sum_d;
        p.sum_kl = a.sum_kl;
        p.best = a.best;
        p.flags = a.flags;
        out[blockIdx.x] = p;
    }
}

constexpr int kMergeThreads = 1024;

__global__ void __launch_bounds__(kMergeThreads)
    audit_pass2(const AuditPartial* __restrict__ parts, int64_t num_parts,
                rlk_audit_result_t* __restrict__ result) {
    Acc a = empty_acc();
    for (int64_t i = threadIdx.x; i < num_parts; i += kMergeThreads) {
        const AuditPartial p = parts[i];
        Acc b;
        b.count = p.count;
        b.arg = p.arg;
        b.sum_d = p.sum_d;
        b.sum_kl = p.sum_kl;
        b.best = p.best;
        b.flags = p.flags;
        merge(a, b);
    }
    a = block_reduce<kMergeThreads>(a);
    if (threadIdx.x == 0) {
        rlk_audit_result_t r;
        r.active_count = a.count;
        r.argmax_index = a.count > 0 ? a.arg : -1;
        r.max_abs_dlogp = a.count > 0 ? a.best : 0.0f;
        r.mean_dlogp = a.sum_d / static_cast<double>(a.count);
        r.approx_kl = a.sum_kl / static_cast<double>(a.count);
        r.error_flags = a.flags;
        *result = r;
    }
}

}  // namespace

// Scratch of rlk_dlogp_audit_noalloc: one partial per 4096-element block for
// up to RLK_AUDIT_NOALLOC_MAX_N tokens (32768 x 40 bytes = 1.25 MiB).  It lives
// in the library image, so every GPU that loads the library holds it until the
// process exits.  Pass 1 writes every slot that pass 2 reads, so nothing in it
// has to start at zero; calls that overlap on the GPU share it and race.
constexpr size_t kNoAllocBlocks = static_cast<size_t>(RLK_AUDIT_NOALLOC_MAX_N) / kAuditBlockElems;
static __device__ __align__(256) AuditPartial g_audit_noalloc_scratch[kNoAllocBlocks];

cudaError_t audit_noalloc_scratch(void** out) {
    // Host code cannot use the array's name as a device address: look the
    // address up once per device, with that device current.
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_audit_noalloc_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *out = addr[dev];
    return cudaSuccess;
}

cudaError_t launch_audit(const float* logp_new, const float* logp_old, const uint8_t* mask,
                         int64_t N, rlk_audit_result_t* result, void* workspace, bool vec_ok,
                         cudaStream_t stream) {
    const size_t blocks = audit_blocks(N);
    AuditPartial* parts = static_cast<AuditPartial*>(workspace);
    if (blocks > 0) {
        if (vec_ok)
            audit_pass1<true><<<static_cast<unsigned>(blocks), kAuditThreads, 0, stream>>>(
                logp_new, logp_old, mask, N, parts);
        else
            audit_pass1<false><<<static_cast<unsigned>(blocks), kAuditThreads, 0, stream>>>(
                logp_new, logp_old, mask, N, parts);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    audit_pass2<<<1, kMergeThreads, 0, stream>>>(parts, static_cast<int64_t>(blocks), result);
    return cudaGetLastError();
}

}  // namespace rlk
