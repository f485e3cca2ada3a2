// audit.cu -- deterministic masked dlogp audit.
//
// "RL-Kernel integration roadmap for vime", Consistency Contract:
// dlogp = recomputed - old; every aggregate over active tokens only;
// max_abs_dlogp is the primary metric, reported with the worst token;
// approx_kl0 = mean(exp(dlogp) - 1 - dlogp); the active-token count.
//
// Pass 1: block b owns the fixed slice [b*4096, (b+1)*4096) (a function of N
// only).  Each thread issues all its loads first (4 float4 of each input and 4
// mask words, streaming cache hint), then handles its 16 elements in ascending
// index order without branches: d = new - old in fp32 (a correctly rounded
// difference), its count, the largest |d| as an order-preserving integer key
// with the first offset attaining it, and fp32 sums of d and of
// kl(d) = exp(d) - 1 - d.  A fixed shuffle tree combines the 32 lanes (fp32
// sums, integer counts), and thread 0 folds the eight warp partials in warp
// order in fp64.  Pass 2: one block merges the per-block partials,
// each thread a fixed strided subset in ascending order, then the same
// fixed tree; it is launched with programmatic dependent launch, so its launch
// overlaps pass 1 and it waits for pass 1's results in-kernel.  No atomics; the
// result is bitwise reproducible for a given N.
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

// Per-thread state of pass 1.  |d| is kept as an order-preserving integer key
// (non-negative floats order like their bit patterns; NaN maps above every
// number), the best key's element offset inside the block, and fp32 sums.
struct ThreadAcc {
    int count = 0;
    uint32_t key = 0;          // 0 = nothing seen (every active |d| has key >= 0 ... see below)
    int arg = -1;              // offset of the best element inside the block
    float sd = 0.f, skl = 0.f;
    uint32_t flags = 0;
};

// key(|d|) + 1, so that 0 means "no active element yet": ties keep the first
// (strict comparison), NaN ranks above +inf.
__device__ __forceinline__ uint32_t abs_key(float d) {
    const uint32_t bits = __float_as_uint(d) & 0x7fffffffu;
    return (bits > 0x7f800000u ? 0x7fc00000u : bits) + 1u;
}

__device__ __forceinline__ void visit3(float nw, float od, uint32_t m, int off, ThreadAcc& a) {
    if (m == 0) return;
    const float d = nw - od;
    const uint32_t key = abs_key(d);
    const bool better = key > a.key;
    a.key = better ? key : a.key;
    a.arg = better ? off : a.arg;
    a.count += 1;
    a.sd += d;
    a.skl += kl_term(d);
    a.flags |= (key > 0x7f800000u) ? 1u : 0u;    // |d| is inf or NaN
}

template <bool VEC>
__global__ void __launch_bounds__(kAuditThreads)
    audit_pass1(const float* __restrict__ nw, const float* __restrict__ od,
                const uint8_t* __restrict__ mask, int64_t N, AuditPartial* __restrict__ out) {
    // let the merge kernel launch now; it waits for this grid before reading
    asm volatile("griddepcontrol.launch_dependents;");
    constexpr int kVec = kAuditV3PerThread / 4;
    constexpr int kBlock = kAuditThreads * kAuditV3PerThread;
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kBlock;
    ThreadAcc a;
    if (VEC && base + kBlock <= N) {
        float4 x[kVec], y[kVec];
        uint32_t m[kVec];
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const int64_t i0 = base + j * (kAuditThreads * 4) + threadIdx.x * 4;
            x[j] = __ldcs(reinterpret_cast<const float4*>(nw + i0));
            y[j] = __ldcs(reinterpret_cast<const float4*>(od + i0));
            m[j] = mask == nullptr ? 0x01010101u
                                   : __ldcs(reinterpret_cast<const unsigned int*>(mask + i0));
        }
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const int o = j * (kAuditThreads * 4) + threadIdx.x * 4;
            visit3(x[j].x, y[j].x, m[j] & 0xffu, o, a);
            visit3(x[j].y, y[j].y, (m[j] >> 8) & 0xffu, o + 1, a);
            visit3(x[j].z, y[j].z, (m[j] >> 16) & 0xffu, o + 2, a);
            visit3(x[j].w, y[j].w, m[j] >> 24, o + 3, a);
        }
    } else {
#pragma unroll 1
        for (int j = 0; j < kVec; ++j) {
            const int o0 = j * (kAuditThreads * 4) + threadIdx.x * 4;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int64_t i = base + o0 + e;
                if (i < N) visit3(nw[i], od[i], mask == nullptr ? 1u : mask[i], o0 + e, a);
            }
        }
    }
    // fixed tree over the warp (fp32 sums, integer counts, key / offset max)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const int c = __shfl_down_sync(0xffffffffu, a.count, off);
        const uint32_t k = __shfl_down_sync(0xffffffffu, a.key, off);
        const int g = __shfl_down_sync(0xffffffffu, a.arg, off);
        const float sd = __shfl_down_sync(0xffffffffu, a.sd, off);
        const float skl = __shfl_down_sync(0xffffffffu, a.skl, off);
        const uint32_t f = __shfl_down_sync(0xffffffffu, a.flags, off);
        if (lane + off < 32) {
            const bool take = k > a.key || (k == a.key && k != 0 && g < a.arg);
            a.key = take ? k : a.key;
            a.arg = take ? g : a.arg;
            a.count += c;
            a.sd += sd;
            a.skl += skl;
            a.flags |= f;
        }
    }
    // the eight warp partials, in warp order, in fp64
    __shared__ Acc warp_acc[kAuditThreads / 32];
    if (lane == 0) {
        Acc w;
        w.count = a.count;
        w.arg = a.key == 0 ? INT64_MAX : base + a.arg;
        w.sum_d = static_cast<double>(a.sd);
        w.sum_kl = static_cast<double>(a.skl);
        w.best = a.key == 0 ? -1.0f : __uint_as_float(a.key - 1u);
        w.flags = a.flags;
        warp_acc[warp] = w;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        Acc t = warp_acc[0];
#pragma unroll
        for (int w = 1; w < kAuditThreads / 32; ++w) merge(t, warp_acc[w]);
        AuditPartial p;
        p.count = t.count;
        p.arg = t.arg;
        p.sum_d = t.sum_d;
        p.sum_kl = t.sum_kl;
        p.best = t.best;
        p.flags = t.flags;
        out[blockIdx.x] = p;
    }
}

constexpr int kMergeThreads = 1024;

__global__ void __launch_bounds__(kMergeThreads)
    audit_pass2(const AuditPartial* __restrict__ parts, int64_t num_parts,
                rlk_audit_result_t* __restrict__ result) {
    // launched early (programmatic dependent launch): wait until every block of
    // pass 1 has finished and its partials are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
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
constexpr size_t kNoAllocBlocks =
    static_cast<size_t>(RLK_AUDIT_NOALLOC_MAX_N) / (kAuditThreads * kAuditV3PerThread);
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
    const size_t blocks = audit_v3_blocks(N);
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
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const AuditPartial* cparts = parts;
    const int64_t nparts = static_cast<int64_t>(blocks);
    return cudaLaunchKernelEx(&cfg, audit_pass2, cparts, nparts, result);
}

}  // namespace rlk
