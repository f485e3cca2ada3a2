// audit.cu -- deterministic masked dlogp audit.
//
// "RL-Kernel integration roadmap for vime", Consistency Contract:
// dlogp = recomputed - old; every aggregate over active tokens only;
// max_abs_dlogp is the primary metric, reported with the worst token;
// approx_kl0 = mean(exp(dlogp) - 1 - dlogp); the active-token count.
//
// Pass 1: the elements are cut into 4096-element slices, and block b owns a
// fixed run of consecutive slices (ceil(slices / 608) of them: a function of N
// only, so that one wave of blocks covers any N).  For each slice a thread
// issues all its loads first (4 float4 of each input and 4 mask words,
// streaming cache hint), then handles its 16 elements without branches:
// d = new - old in fp32 (a correctly rounded difference), its count, the
// largest |d| as an order-preserving integer key with the first offset
// attaining it, and fp32 sums of d and of kl(d) = exp(d) - 1 - d, in four
// interleaved chains merged in a fixed order; each slice's sums are added to
// the thread's float-pair sums (about 48 bits: two-sum; this GPU's fp64 units
// are few and slow).  A fixed shuffle tree combines the 32 lanes, and thread 0
// folds the eight warp partials in warp order.  Pass 2: one block merges
// the per-block partials,
// each thread a fixed strided subset in ascending order, then the same
// fixed tree; it is launched with programmatic dependent launch, so its launch
// overlaps pass 1 and it waits for pass 1's results in-kernel.  No atomics; the
// result is bitwise reproducible for a given N.
//
// kl(d) for |d| < 1/2 is the Taylor series d^2 (1/2 + d/6 + d^2/24 + ...)
// through the d^9 term (truncation below 3e-9 relative); elsewhere it is
// expm1f(d) - d, where no cancellation arises.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "rlk_internal.h"

namespace rlk {

namespace {

// exp(d) - 1 - d for |d| < 1/16: the Taylor series to d^6 (truncation below 4e-10
// relative).  Branch-free, so the audit's fast path evaluates it for every element.
__device__ __forceinline__ float kl_small(float d) {
    float p = 1.0f / 720.0f;
    p = fmaf(p, d, 1.0f / 120.0f);
    p = fmaf(p, d, 1.0f / 24.0f);
    p = fmaf(p, d, 1.0f / 6.0f);
    p = fmaf(p, d, 0.5f);
    return d * d * p;
}

__device__ __forceinline__ float kl_term(float d) {
    if (fabsf(d) < 0.0625f) return kl_small(d);
    if (fabsf(d) < 0.5f) {             // to d^9: truncation below 3e-8 relative
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

// a + b as a float pair (two-sum, then renormalisation), in a fixed
// evaluation order: deterministic, and exact to about 2^-44 relative.
__device__ __forceinline__ DFloat df_add(DFloat a, DFloat b) {
    const float s = __fadd_rn(a.hi, b.hi);
    const float bv = __fsub_rn(s, a.hi);
    const float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bv)), __fsub_rn(b.hi, bv));
    const float lo = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
    const float hi = __fadd_rn(s, lo);
    return DFloat{hi, __fsub_rn(lo, __fsub_rn(hi, s))};
}

__device__ __forceinline__ double df_value(DFloat a) {
    return static_cast<double>(a.hi) + static_cast<double>(a.lo);
}

struct Acc {
    int64_t count;
    int64_t arg;
    DFloat sum_d;
    DFloat sum_kl;
    float best;
    uint32_t flags;
};

__device__ __forceinline__ Acc empty_acc() {
    Acc a;
    a.count = 0;
    a.arg = INT64_MAX;
    a.sum_d = DFloat{0.f, 0.f};
    a.sum_kl = DFloat{0.f, 0.f};
    a.best = -1.0f;
    a.flags = 0;
    return a;
}

// a := a (+) b, with a covering lower indices than b
__device__ __forceinline__ void merge(Acc& a, const Acc& b) {
    a.count += b.count;
    a.sum_d = df_add(a.sum_d, b.sum_d);
    a.sum_kl = df_add(a.sum_kl, b.sum_kl);
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
    b.sum_d.hi = __shfl_down_sync(0xffffffffu, a.sum_d.hi, off);
    b.sum_d.lo = __shfl_down_sync(0xffffffffu, a.sum_d.lo, off);
    b.sum_kl.hi = __shfl_down_sync(0xffffffffu, a.sum_kl.hi, off);
    b.sum_kl.lo = __shfl_down_sync(0xffffffffu, a.sum_kl.lo, off);
    b.best = __shfl_down_sync(0xffffffffu, a.best, off);
    b.flags = __shfl_down_sync(0xffffffffu, a.flags, off);
    return b;
}

// Barrier 1 over the first `threads` threads of the block (the audit kernels'
// reducing threads; a streaming kernel's copy warp does not take part).
__device__ __forceinline__ void named_barrier(int threads) {
    asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory");
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
    named_barrier(THREADS);
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

// number of nonzero bytes in a word of four mask bytes
__device__ __forceinline__ int active_bytes(uint32_t m) {
    const uint32_t hi = ((m & 0x7f7f7f7fu) + 0x7f7f7f7fu) | m;
    return __popc(hi & 0x80808080u);
}

// Pass 1's partition is a function of N only: slices of 4096 elements, dealt out
// round-robin to G = min(slices, kAuditMaxBlocks) blocks (block b takes slices b,
// b + G, b + 2G, ... in ascending order), so that one wave of blocks covers any N
// (608 = 4 resident blocks on each of 152 SMs), the whole grid sweeps the inputs
// front to back together, and the merge reads at most kAuditMaxBlocks partials.
constexpr int64_t kAuditMaxBlocks = 608;
constexpr int kSlice = kAuditThreads * kAuditV3PerThread;   // 4096 elements
constexpr int kVec = kAuditV3PerThread / 4;                 // float4 groups per thread

inline int64_t audit_pass1_blocks(int64_t N) {
    const int64_t slices = static_cast<int64_t>(audit_v3_blocks(N));
    return slices < kAuditMaxBlocks ? slices : kAuditMaxBlocks;
}

// The order-preserving key of |d| as the running max compares it: the bits of |d|
// with every NaN mapped to one pattern above inf, plus one, so that 0 means "no
// active element" (ties keep the first offset: strict comparison).
__device__ __forceinline__ uint32_t key_of_bits(uint32_t b) {
    return (b > 0x7f800000u ? 0x7fc00000u : b) + 1u;
}

// One slice seen by one thread: its elements j*1024 + 4*tid + e (group j, lane e of
// the group) with the new and old values and the four mask bytes of each group.
// An inactive element contributes d = 0 to the sums and nothing to the running max.
// The per-element work is branch-free and short: the sums of d and of
// kl(d) = exp(d) - 1 - d (its small-|d| series; one accumulator per group, so the
// four groups' dependency chains interleave, merged in a fixed tree) and the largest
// |d| bits of each group.  Two things are done per slice, not per element: when some
// |d| reaches 1/16 (or is inf / NaN) the slice's kl sums are formed again with the
// exact kl_term; and the offset of the slice's largest |d| (the first one, in element
// order, on ties) is looked up only when that value beats `best_key`, the thread's
// running best, since otherwise it is not needed.  a.key is the slice's key, a.arg
// its first offset when a.key > best_key.
__device__ __forceinline__ void visit_slice(const float4 (&x)[kVec], const float4 (&y)[kVec],
                                            const uint32_t (&m)[kVec], int tid, uint32_t best_key,
                                            ThreadAcc& a) {
    float sd[kVec], skl[kVec];
    uint32_t gmax[kVec];
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        a.count += active_bytes(m[j]);
        const float xs[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
        const float ys[4] = {y[j].x, y[j].y, y[j].z, y[j].w};
        sd[j] = 0.f;
        skl[j] = 0.f;
        gmax[j] = 0u;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const bool act = ((m[j] >> (8 * e)) & 0xffu) != 0u;
            const float d = act ? xs[e] - ys[e] : 0.f;
            gmax[j] = max(gmax[j], __float_as_uint(d) & 0x7fffffffu);
            sd[j] += d;
            skl[j] += kl_small(d);
        }
    }
    const uint32_t smax = max(max(gmax[0], gmax[1]), max(gmax[2], gmax[3]));
    // an inf or NaN |d| exists exactly when the largest bits reach those of inf
    a.flags = smax >= 0x7f800000u ? 1u : 0u;
    if (smax >= 0x3d800000u) {                 // some |d| >= 1/16, inf or NaN: exact terms
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const float xs[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
            const float ys[4] = {y[j].x, y[j].y, y[j].z, y[j].w};
            skl[j] = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool act = ((m[j] >> (8 * e)) & 0xffu) != 0u;
                skl[j] += act ? kl_term(xs[e] - ys[e]) : 0.f;
            }
        }
    }
    static_assert(kVec == 4, "the fixed summation tree below assumes four groups");
    a.sd = (sd[0] + sd[1]) + (sd[2] + sd[3]);
    a.skl = (skl[0] + skl[1]) + (skl[2] + skl[3]);
    a.key = a.count > 0 ? key_of_bits(smax) : 0u;
    a.arg = -1;
    if (a.key > best_key) {
        // the first active element, in (group, lane) order, whose key is the slice's
        int arg = -1;
#pragma unroll
        for (int j = kVec - 1; j >= 0; --j) {
            const float xs[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
            const float ys[4] = {y[j].x, y[j].y, y[j].z, y[j].w};
#pragma unroll
            for (int e = 3; e >= 0; --e) {
                const bool act = ((m[j] >> (8 * e)) & 0xffu) != 0u;
                const uint32_t b = __float_as_uint(xs[e] - ys[e]) & 0x7fffffffu;
                arg = (act && key_of_bits(b) == a.key) ? j * (kAuditThreads * 4) + tid * 4 + e
                                                       : arg;
            }
        }
        a.arg = arg;
    }
}

// A slice read straight from global memory: vector loads when VEC (16-byte aligned
// inputs, whole slice inside N), else element by element with elements past N
// inactive.  Either way the arithmetic is visit_slice's.
template <bool VEC>
__device__ __forceinline__ void load_and_visit_slice(const float* nw, const float* od,
                                                     const uint8_t* mask, int64_t N,
                                                     int64_t base, uint32_t best_key,
                                                     ThreadAcc& a) {
    float4 x[kVec], y[kVec];
    uint32_t m[kVec];
    if (VEC && base + kSlice <= N) {
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const int64_t i0 = base + j * (kAuditThreads * 4) + threadIdx.x * 4;
            x[j] = __ldcs(reinterpret_cast<const float4*>(nw + i0));
            y[j] = __ldcs(reinterpret_cast<const float4*>(od + i0));
            m[j] = mask == nullptr ? 0x01010101u
                                   : __ldcs(reinterpret_cast<const unsigned int*>(mask + i0));
        }
    } else {
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const int64_t i0 = base + j * (kAuditThreads * 4) + threadIdx.x * 4;
            float xv[4], yv[4];
            uint32_t mv = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool in = i0 + e < N;
                xv[e] = in ? nw[i0 + e] : 0.f;
                yv[e] = in ? od[i0 + e] : 0.f;
                const uint32_t b = in ? (mask == nullptr ? 1u : (mask[i0 + e] != 0 ? 1u : 0u)) : 0u;
                mv |= b << (8 * e);
            }
            x[j] = make_float4(xv[0], xv[1], xv[2], xv[3]);
            y[j] = make_float4(yv[0], yv[1], yv[2], yv[3]);
            m[j] = mv;
        }
    }
    visit_slice(x, y, m, threadIdx.x, best_key, a);
}

// The running state of a block's thread over the block's slices, visited in ascending
// order: count, the best key and its element index (strictly greater replaces, so the
// first index wins ties), float-pair sums of each slice's fp32 sums.
struct RunAcc {
    int count = 0;
    uint32_t best_key = 0;
    int64_t best_off = -1;
    uint32_t flags = 0;
    DFloat sum_d{0.f, 0.f}, sum_kl{0.f, 0.f};

    __device__ __forceinline__ void add_slice(const ThreadAcc& a, int64_t slice_base) {
        count += a.count;
        if (a.key > best_key) {
            best_key = a.key;
            best_off = slice_base + a.arg;
        }
        flags |= a.flags;
        sum_d = df_add(sum_d, DFloat{a.sd, 0.f});
        sum_kl = df_add(sum_kl, DFloat{a.skl, 0.f});
    }
};

// The block's partial from its kAuditThreads threads: a fixed tree over each
// warp (float-pair sums, integer counts, key / index max), then the eight warp
// partials in warp order, written by thread 0.
__device__ __forceinline__ void finish_block(RunAcc r, AuditPartial* out) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const int c = __shfl_down_sync(0xffffffffu, r.count, off);
        const uint32_t k = __shfl_down_sync(0xffffffffu, r.best_key, off);
        const int64_t g = __shfl_down_sync(0xffffffffu, r.best_off, off);
        DFloat sd, skl;
        sd.hi = __shfl_down_sync(0xffffffffu, r.sum_d.hi, off);
        sd.lo = __shfl_down_sync(0xffffffffu, r.sum_d.lo, off);
        skl.hi = __shfl_down_sync(0xffffffffu, r.sum_kl.hi, off);
        skl.lo = __shfl_down_sync(0xffffffffu, r.sum_kl.lo, off);
        const uint32_t f = __shfl_down_sync(0xffffffffu, r.flags, off);
        if (lane + off < 32) {
            const bool take = k > r.best_key || (k == r.best_key && k != 0 && g < r.best_off);
            r.best_key = take ? k : r.best_key;
            r.best_off = take ? g : r.best_off;
            r.count += c;
            r.sum_d = df_add(r.sum_d, sd);
            r.sum_kl = df_add(r.sum_kl, skl);
            r.flags |= f;
        }
    }
    __shared__ Acc warp_acc[kAuditThreads / 32];
    if (lane == 0) {
        Acc w;
        w.count = r.count;
        w.arg = r.best_key == 0 ? INT64_MAX : r.best_off;
        w.sum_d = r.sum_d;
        w.sum_kl = r.sum_kl;
        w.best = r.best_key == 0 ? -1.0f : __uint_as_float(r.best_key - 1u);
        w.flags = r.flags;
        warp_acc[warp] = w;
    }
    named_barrier(kAuditThreads);
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

// Pass 1 (any alignment; vector loads when VEC); a second launch merges.
template <bool VEC>
__global__ void __launch_bounds__(kAuditThreads)
    audit_pass1(const float* __restrict__ nw, const float* __restrict__ od,
                const uint8_t* __restrict__ mask, int64_t N, AuditPartial* __restrict__ out) {
    // let the merge kernel launch now; it waits for this grid before reading
    asm volatile("griddepcontrol.launch_dependents;");
    const int64_t slices = (N + kSlice - 1) / kSlice;
    RunAcc r;
#pragma unroll 1
    for (int64_t sl = blockIdx.x; sl < slices; sl += gridDim.x) {
        ThreadAcc a;
        load_and_visit_slice<VEC>(nw, od, mask, N, sl * kSlice, r.best_key, a);
        r.add_slice(a, sl * kSlice);
    }
    finish_block(r, out);
}

constexpr int kMergeThreads = 1024;
constexpr int kMergeBatch = 4;   // partials a merge thread loads before it folds them

__device__ __forceinline__ Acc to_acc(const AuditPartial& p) {
    Acc b;
    b.count = p.count;
    b.arg = p.arg;
    b.sum_d = p.sum_d;
    b.sum_kl = p.sum_kl;
    b.best = p.best;
    b.flags = p.flags;
    return b;
}

// Thread t folds partials t, t + THREADS, t + 2 THREADS, ... in ascending order (they
// are loaded kMergeBatch at a time so that the loads overlap; the order is unchanged),
// then the fixed block tree; thread 0 writes the result.
template <int THREADS>
__device__ void merge_partials(const AuditPartial* parts, int64_t num_parts,
                               rlk_audit_result_t* result) {
    Acc a = empty_acc();
    int64_t i = threadIdx.x;
    for (; i + (kMergeBatch - 1) * THREADS < num_parts; i += kMergeBatch * THREADS) {
        AuditPartial p[kMergeBatch];
#pragma unroll
        for (int j = 0; j < kMergeBatch; ++j) p[j] = parts[i + j * THREADS];
#pragma unroll
        for (int j = 0; j < kMergeBatch; ++j) merge(a, to_acc(p[j]));
    }
    for (; i < num_parts; i += THREADS) merge(a, to_acc(parts[i]));
    a = block_reduce<THREADS>(a);
    if (threadIdx.x == 0) {
        rlk_audit_result_t r;
        r.active_count = a.count;
        r.argmax_index = a.count > 0 ? a.arg : -1;
        r.max_abs_dlogp = a.count > 0 ? a.best : 0.0f;
        r.mean_dlogp = df_value(a.sum_d) / static_cast<double>(a.count);
        r.approx_kl = df_value(a.sum_kl) / static_cast<double>(a.count);
        r.error_flags = a.flags;
        *result = r;
    }
}

__global__ void __launch_bounds__(kMergeThreads)
    audit_pass2(const AuditPartial* __restrict__ parts, int64_t num_parts,
                rlk_audit_result_t* __restrict__ result) {
    // launched early (programmatic dependent launch): wait until every block of
    // pass 1 has finished and its partials are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    merge_partials<kMergeThreads>(parts, num_parts, result);
}

// ----------------------------------------------------------------------------- extended audit
//
// The consistency contract's minimum diagnostics beyond the base audit: mean
// |d|, mean ratio0 = exp(d), clipfrac0 = #{|exp(d) - 1| > eps} / count, the
// p50 / p90 / p99 of |d| by the nearest-rank rule (1-based rank
// ceil(p * count) of the ascending order), and the worst token's sequence and
// position.  Pass 1 is the base pass plus three more per-thread sums; the
// percentiles are selected exactly by a three-pass radix select over the
// order-preserving 32-bit key of |d| (digits of 11, 11 and 10 bits), with
// integer histograms: the counts, hence the selected values, are exact and
// reproducible however the atomics interleave.

struct ExtPartial {
    AuditPartial base;
    DFloat sum_abs, sum_ratio;
    int64_t clip;
};

// One active element of the extended pass: the base audit's terms, its |d| key,
// and the sums of |d|, of the ratio exp(d) and the count of clipped ratios.
__device__ __forceinline__ uint32_t visit_ext(float nv, float ov, int off, float eps,
                                              ThreadAcc& a, float& sabs, float& sratio,
                                              int& clip) {
    visit3(nv, ov, 1u, off, a);
    const float d = nv - ov;
    const float r = expf(d);
    sabs += fabsf(d);
    sratio += r;
    clip += fabsf(r - 1.0f) > eps ? 1 : 0;
    return abs_key(d);
}

struct SelectState {
    uint32_t prefix[3];
    uint32_t pad;
    int64_t rank[3];
};

constexpr int kHistBins = 2048;
constexpr int kHistBlocksPerSm = 8;

template <bool VEC>
__global__ void __launch_bounds__(kAuditThreads)
    audit_ext_pass1(const float* __restrict__ nw, const float* __restrict__ od,
                    const uint8_t* __restrict__ mask, int64_t N, float eps,
                    ExtPartial* __restrict__ out, uint32_t* __restrict__ keys) {
    constexpr int kBlock = kAuditThreads * kAuditV3PerThread;
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kBlock;
    ThreadAcc a;
    float sabs = 0.f, sratio = 0.f;
    int clip = 0;
    constexpr int kVec = kAuditV3PerThread / 4;
    if (VEC && base + kBlock <= N) {
        // every load first (4 float4 of each input, 4 mask words), then the elements
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
            const int o0 = j * (kAuditThreads * 4) + threadIdx.x * 4;
            const float xs[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
            const float ys[4] = {y[j].x, y[j].y, y[j].z, y[j].w};
            uint32_t k4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                k4[e] = ((m[j] >> (8 * e)) & 0xffu) != 0u
                            ? visit_ext(xs[e], ys[e], o0 + e, eps, a, sabs, sratio, clip)
                            : 0u;
            // |d| keys for the percentile passes (0 for inactive tokens)
            *reinterpret_cast<uint4*>(keys + base + o0) = make_uint4(k4[0], k4[1], k4[2], k4[3]);
        }
    } else {
#pragma unroll 1
        for (int j = 0; j < kVec; ++j) {
            const int o0 = j * (kAuditThreads * 4) + threadIdx.x * 4;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int64_t i = base + o0 + e;
                if (i >= N) continue;
                const bool act = mask == nullptr || mask[i] != 0;
                keys[i] = act ? visit_ext(nw[i], od[i], o0 + e, eps, a, sabs, sratio, clip) : 0u;
            }
        }
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const int c = __shfl_down_sync(0xffffffffu, a.count, off);
        const uint32_t k = __shfl_down_sync(0xffffffffu, a.key, off);
        const int g = __shfl_down_sync(0xffffffffu, a.arg, off);
        const float sd = __shfl_down_sync(0xffffffffu, a.sd, off);
        const float skl = __shfl_down_sync(0xffffffffu, a.skl, off);
        const uint32_t f = __shfl_down_sync(0xffffffffu, a.flags, off);
        const float sa = __shfl_down_sync(0xffffffffu, sabs, off);
        const float sr = __shfl_down_sync(0xffffffffu, sratio, off);
        const int cl = __shfl_down_sync(0xffffffffu, clip, off);
        if (lane + off < 32) {
            const bool take = k > a.key || (k == a.key && k != 0 && g < a.arg);
            a.key = take ? k : a.key;
            a.arg = take ? g : a.arg;
            a.count += c;
            a.sd += sd;
            a.skl += skl;
            a.flags |= f;
            sabs += sa;
            sratio += sr;
            clip += cl;
        }
    }
    __shared__ Acc warp_acc[kAuditThreads / 32];
    __shared__ float warp_abs[kAuditThreads / 32], warp_ratio[kAuditThreads / 32];
    __shared__ int warp_clip[kAuditThreads / 32];
    if (lane == 0) {
        Acc w;
        w.count = a.count;
        w.arg = a.key == 0 ? INT64_MAX : base + a.arg;
        w.sum_d = DFloat{a.sd, 0.f};
        w.sum_kl = DFloat{a.skl, 0.f};
        w.best = a.key == 0 ? -1.0f : __uint_as_float(a.key - 1u);
        w.flags = a.flags;
        warp_acc[warp] = w;
        warp_abs[warp] = sabs;
        warp_ratio[warp] = sratio;
        warp_clip[warp] = clip;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        Acc t = warp_acc[0];
        DFloat sa{warp_abs[0], 0.f}, sr{warp_ratio[0], 0.f};
        int64_t cl = warp_clip[0];
#pragma unroll
        for (int w = 1; w < kAuditThreads / 32; ++w) {
            merge(t, warp_acc[w]);
            sa = df_add(sa, DFloat{warp_abs[w], 0.f});
            sr = df_add(sr, DFloat{warp_ratio[w], 0.f});
            cl += warp_clip[w];
        }
        ExtPartial p;
        p.base.count = t.count;
        p.base.arg = t.arg;
        p.base.sum_d = t.sum_d;
        p.base.sum_kl = t.sum_kl;
        p.base.best = t.best;
        p.base.flags = t.flags;
        p.sum_abs = sa;
        p.sum_ratio = sr;
        p.clip = cl;
        out[blockIdx.x] = p;
    }
}

// One block: fixed-order merge of the partials; writes the sums into the
// result, the nearest ranks into the select state, clears the histograms.
__global__ void __launch_bounds__(kMergeThreads)
    audit_ext_merge(const ExtPartial* __restrict__ parts, int64_t num_parts,
                    const int64_t* __restrict__ seq_offsets, int64_t num_seqs,
                    rlk_audit_ext_t* __restrict__ result, SelectState* __restrict__ sel,
                    uint32_t* __restrict__ hist) {
    Acc a = empty_acc();
    DFloat sa{0.f, 0.f}, sr{0.f, 0.f};
    int64_t cl = 0;
    // ascending partials per thread, loaded in batches (as in the base audit's merge)
    auto fold = [&](const ExtPartial& p) {
        merge(a, to_acc(p.base));
        sa = df_add(sa, p.sum_abs);
        sr = df_add(sr, p.sum_ratio);
        cl += p.clip;
    };
    int64_t i = threadIdx.x;
    for (; i + (kMergeBatch - 1) * kMergeThreads < num_parts; i += kMergeBatch * kMergeThreads) {
        ExtPartial p[kMergeBatch];
#pragma unroll
        for (int j = 0; j < kMergeBatch; ++j) p[j] = parts[i + j * kMergeThreads];
#pragma unroll
        for (int j = 0; j < kMergeBatch; ++j) fold(p[j]);
    }
    for (; i < num_parts; i += kMergeThreads) fold(parts[i]);
    for (int i = threadIdx.x; i < 3 * kHistBins; i += kMergeThreads) hist[i] = 0u;
    a = block_reduce<kMergeThreads>(a);
    __shared__ DFloat s_abs[kMergeThreads / 32], s_ratio[kMergeThreads / 32];
    __shared__ long long s_clip[kMergeThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // the same fixed tree for the three extra sums
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        DFloat x, y;
        x.hi = __shfl_down_sync(0xffffffffu, sa.hi, off);
        x.lo = __shfl_down_sync(0xffffffffu, sa.lo, off);
        y.hi = __shfl_down_sync(0xffffffffu, sr.hi, off);
        y.lo = __shfl_down_sync(0xffffffffu, sr.lo, off);
        const long long z = __shfl_down_sync(0xffffffffu, static_cast<long long>(cl), off);
        if (lane + off < 32) {
            sa = df_add(sa, x);
            sr = df_add(sr, y);
            cl += z;
        }
    }
    if (lane == 0) {
        s_abs[warp] = sa;
        s_ratio[warp] = sr;
        s_clip[warp] = cl;
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    for (int w = 1; w < kMergeThreads / 32; ++w) {
        s_abs[0] = df_add(s_abs[0], s_abs[w]);
        s_ratio[0] = df_add(s_ratio[0], s_ratio[w]);
        s_clip[0] += s_clip[w];
    }
    rlk_audit_ext_t r;
    r.active_count = a.count;
    r.argmax_index = a.count > 0 ? a.arg : -1;
    r.argmax_seq = -1;
    r.argmax_pos = -1;
    if (seq_offsets != nullptr && num_seqs > 0 && a.count > 0) {
        int64_t lo = 0, hi = num_seqs;      // last s < num_seqs with seq_offsets[s] <= arg
        while (hi - lo > 1) {
            const int64_t mid = (lo + hi) >> 1;
            if (seq_offsets[mid] <= a.arg) lo = mid; else hi = mid;
        }
        if (a.arg >= seq_offsets[lo] && a.arg < seq_offsets[lo + 1]) {
            r.argmax_seq = lo;
            r.argmax_pos = a.arg - seq_offsets[lo];
        }
    }
    r.clip_count = s_clip[0];
    const double cnt = static_cast<double>(a.count);
    r.mean_dlogp = df_value(a.sum_d) / cnt;
    r.mean_abs_dlogp = df_value(s_abs[0]) / cnt;
    r.mean_ratio = df_value(s_ratio[0]) / cnt;
    r.approx_kl = df_value(a.sum_kl) / cnt;
    r.max_abs_dlogp = a.count > 0 ? a.best : 0.0f;
    r.p50_abs_dlogp = r.p90_abs_dlogp = r.p99_abs_dlogp = __int_as_float(0x7fc00000);
    r.clipfrac = static_cast<float>(static_cast<double>(s_clip[0]) / cnt);
    r.error_flags = a.flags;
    *result = r;
    const int pct[3] = {50, 90, 99};
    for (int q = 0; q < 3; ++q) {
        sel->prefix[q] = 0u;
        sel->rank[q] = (pct[q] * a.count + 99) / 100;   // nearest rank, 1-based (0 if none)
    }
}

// Histogram of one digit of the |d| keys of the active elements that match
// each percentile's prefix so far.
// One radix-select pass over the |d| keys written by pass 1 (0 = inactive).
// Pass 0 (top 11 bits) is the same for the three percentiles, so it builds a
// single histogram; lanes of a warp that hit the same bin add their count with
// one shared-memory atomic (|d| concentrates in few bins).  Passes 1 and 2
// count, per percentile, the keys whose higher digits match its prefix.
// Blocks stride over the 4096-key slices (a grid of a few blocks per SM), so
// a block adds its shared histogram into the global one once for many slices;
// the counts are integers, so the totals do not depend on the grid.  Pass 0
// gives each warp its own copy of the histogram (the few hot bins would
// otherwise serialise the warps' atomics) and sums the copies at the end.
template <int PASS>
__host__ __device__ constexpr int hist_copies() {
    return PASS == 0 ? kAuditThreads / 32 : 3;
}

template <int PASS>
__host__ __device__ constexpr size_t hist_smem_bytes() {
    return static_cast<size_t>(hist_copies<PASS>()) * kHistBins * 4;
}

template <int PASS>
__global__ void __launch_bounds__(kAuditThreads)
    audit_ext_hist(const uint32_t* __restrict__ keys, int64_t N, int64_t num_slices,
                   const SelectState* __restrict__ sel, uint32_t* __restrict__ hist) {
    constexpr int kShift = PASS == 0 ? 21 : (PASS == 1 ? 10 : 0);
    constexpr uint32_t kDigitMask = PASS == 2 ? 0x3ffu : 0x7ffu;
    constexpr int kPrefixShift = PASS == 1 ? 21 : 10;
    constexpr int kHists = PASS == 0 ? 1 : 3;
    constexpr int kCopies = hist_copies<PASS>();
    extern __shared__ uint32_t h[];                 // [kCopies][kHistBins]
    for (int i = threadIdx.x; i < kCopies * kHistBins; i += kAuditThreads) h[i] = 0u;
    uint32_t* hw = h + (PASS == 0 ? (threadIdx.x >> 5) * kHistBins : 0);   // this warp's copy
    uint32_t pre[3];
    bool want[3];
#pragma unroll
    for (int q = 0; q < 3; ++q) {
        pre[q] = sel->prefix[q];
        want[q] = sel->rank[q] > 0;
    }
    __syncthreads();
    for (int64_t slice = blockIdx.x; slice < num_slices && (PASS > 0 || want[0] || want[1] ||
                                                            want[2]);
         slice += gridDim.x) {
        constexpr int kBlock = kAuditThreads * kAuditV3PerThread;
        const int64_t base = slice * kBlock;
        const int lane = threadIdx.x & 31;
        constexpr int kVec = kAuditV3PerThread / 4;
        uint32_t k[kVec][4];
        // every load first, then the counting (the atomics would otherwise keep the
        // compiler from moving later loads ahead)
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const int64_t i0 = base + j * (kAuditThreads * 4) + threadIdx.x * 4;
            if (i0 + 4 <= N) {
                const uint4 v = __ldcs(reinterpret_cast<const uint4*>(keys + i0));
                k[j][0] = v.x;
                k[j][1] = v.y;
                k[j][2] = v.z;
                k[j][3] = v.w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) k[j][e] = i0 + e < N ? keys[i0 + e] : 0u;
            }
        }
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t key = k[j][e];
                const uint32_t digit = (key >> kShift) & kDigitMask;
                if (PASS == 0) {
                    // every lane reaches this point: aggregate equal bins across the warp
                    const unsigned valid = __ballot_sync(0xffffffffu, key != 0u);
                    if (key != 0u) {
                        const unsigned peers = __match_any_sync(valid, digit);
                        if (lane == __ffs(peers) - 1) atomicAdd(&hw[digit], __popc(peers));
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 3; ++q)
                        if (key != 0u && want[q] && (key >> kPrefixShift) == pre[q])
                            atomicAdd(&h[q * kHistBins + digit], 1u);
                }
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kHists * kHistBins; i += kAuditThreads) {
        uint32_t c = h[i];
        if constexpr (PASS == 0) {
#pragma unroll
            for (int w = 1; w < kCopies; ++w) c += h[w * kHistBins + i];
        }
        if (c != 0u) atomicAdd(&hist[i], c);
    }
}

// Picks, for each percentile, the bin holding its rank; extends the prefix by
// that digit and clears the histogram for the next pass.  After the last pass
// the prefix is the selected key, written to the result.  Each of the 256
// threads owns a run of consecutive bins; an exclusive scan of the runs' counts
// (integers, so exact) tells the one thread whose run holds the rank, and that
// thread walks its own run.
constexpr int kSelectThreads = 256;

template <int PASS>
__global__ void __launch_bounds__(kSelectThreads)
    audit_ext_select(SelectState* __restrict__ sel, uint32_t* __restrict__ hist,
                     rlk_audit_ext_t* __restrict__ result) {
    constexpr int kBits = PASS == 2 ? 10 : 11;
    constexpr int kRun = (1 << kBits) / kSelectThreads;     // 8 bins (4 in the last pass)
    __shared__ int64_t warp_sum[kSelectThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int q = 0; q < 3; ++q) {
        const int64_t rank = sel->rank[q];           // the same for every thread
        if (rank <= 0) continue;
        const uint32_t* hq = hist + (PASS == 0 ? 0 : q * kHistBins) + threadIdx.x * kRun;
        uint32_t c[kRun];
        int64_t run = 0;
#pragma unroll
        for (int j = 0; j < kRun; ++j) {
            c[j] = hq[j];
            run += c[j];
        }
        // inclusive scan over the block: lanes, then warps in order
        int64_t incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int64_t o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) warp_sum[warp] = incl;
        __syncthreads();
        int64_t before = 0;
        for (int w = 0; w < warp; ++w) before += warp_sum[w];
        const int64_t excl = before + incl - run;
        if (excl < rank && rank <= excl + run) {
            int64_t cum = excl;                      // count below the selected bin
            int bin = -1;
#pragma unroll
            for (int j = 0; j < kRun; ++j) {
                if (bin < 0) {
                    if (rank <= cum + c[j])
                        bin = j;
                    else
                        cum += c[j];
                }
            }
            const uint32_t digit = static_cast<uint32_t>(threadIdx.x * kRun + bin);
            sel->rank[q] = rank - cum;
            sel->prefix[q] = (sel->prefix[q] << kBits) | digit;
            if (PASS == 2) {
                const float v = __uint_as_float(sel->prefix[q] - 1u);
                if (q == 0) result->p50_abs_dlogp = v;
                if (q == 1) result->p90_abs_dlogp = v;
                if (q == 2) result->p99_abs_dlogp = v;
            }
        }
        __syncthreads();                             // warp_sum is reused for the next q
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 3 * kHistBins; i += kSelectThreads) hist[i] = 0u;
}

}  // namespace

// Scratch of rlk_dlogp_audit_noalloc: room for the partials of pass 1 (it writes
// at most kAuditMaxBlocks of them, whatever N).  It lives in the library image, so
// every GPU that loads the library holds it until the process exits.  Pass 1 writes
// every partial that the merge reads, so nothing in it has to start at zero; calls
// that overlap on the GPU share it and race.
constexpr size_t kNoAllocBlocks =
    static_cast<size_t>(RLK_AUDIT_NOALLOC_MAX_N) / (kAuditThreads * kAuditV3PerThread);
static_assert(kNoAllocBlocks >= static_cast<size_t>(kAuditMaxBlocks),
              "the no-alloc scratch must hold every partial pass 1 can write");
static __device__ __align__(256) AuditPartial g_audit_noalloc_scratch[kNoAllocBlocks];

namespace {

using PfnCtxGetCurrent = CUresult (*)(CUcontext*);
using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long*);

template <class F>
F driver_fn(const char* name) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<F>(p);
}

}  // namespace

cudaError_t audit_noalloc_scratch(void** parts) {
    // Host code cannot use the array's name as a device address: the address is looked
    // up with the device current, and cached per device together with the unique id of
    // the context it belongs to, so that a context created anew (after cudaDeviceReset,
    // say) is looked up again instead of reusing a stale address.
    static std::mutex mu;
    static std::once_flag once;
    static PfnCtxGetCurrent get_current = nullptr;
    static PfnCtxGetId get_id = nullptr;
    static void* addr[64] = {};
    static unsigned long long ctx_id[64] = {};
    std::call_once(once, [] {
        get_current = driver_fn<PfnCtxGetCurrent>("cuCtxGetCurrent");
        get_id = driver_fn<PfnCtxGetId>("cuCtxGetId");
    });
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    // without a current context yet (no id), the address is looked up on every call
    unsigned long long id = 0;
    CUcontext ctx = nullptr;
    const bool have_id = get_current != nullptr && get_id != nullptr &&
                         get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
                         get_id(ctx, &id) == CUDA_SUCCESS;
    std::lock_guard<std::mutex> lock(mu);
    if (!have_id || addr[dev] == nullptr || ctx_id[dev] != id) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_audit_noalloc_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
        ctx_id[dev] = have_id ? id : 0;
    }
    *parts = addr[dev];
    return cudaSuccess;
}

// Pass 1 (vector loads when vec_ok, element loads otherwise: the same arithmetic),
// then one block that merges, launched by programmatic dependent launch so that its
// launch overlaps pass 1.
cudaError_t launch_audit(const float* logp_new, const float* logp_old, const uint8_t* mask,
                         int64_t N, rlk_audit_result_t* result, void* partials, bool vec_ok,
                         cudaStream_t stream) {
    AuditPartial* parts = static_cast<AuditPartial*>(partials);
    const unsigned blocks = static_cast<unsigned>(audit_pass1_blocks(N));
    if (blocks > 0) {
        if (vec_ok)
            audit_pass1<true><<<blocks, kAuditThreads, 0, stream>>>(logp_new, logp_old, mask, N,
                                                                    parts);
        else
            audit_pass1<false><<<blocks, kAuditThreads, 0, stream>>>(logp_new, logp_old, mask, N,
                                                                     parts);
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

// partials | 3 histograms | select state | |d| keys [N] (uint32)
static size_t ext_keys_off(int64_t N) {
    return align_up(align_up(audit_v3_blocks(N) * sizeof(ExtPartial), 256) + 3 * kHistBins * 4 +
                    sizeof(SelectState), 256);
}

size_t audit_ext_workspace(int64_t N) {
    return ext_keys_off(N) + align_up(static_cast<size_t>(N) * 4, 256) + 256;
}

cudaError_t launch_audit_ext(const float* logp_new, const float* logp_old, const uint8_t* mask,
                             int64_t N, const int64_t* seq_offsets, int64_t num_seqs, float eps,
                             rlk_audit_ext_t* result, void* workspace, bool vec_ok, int sms,
                             cudaStream_t stream) {
    const size_t blocks = audit_v3_blocks(N);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    ExtPartial* parts = reinterpret_cast<ExtPartial*>(ws);
    uint32_t* hist = reinterpret_cast<uint32_t*>(ws + align_up(blocks * sizeof(ExtPartial), 256));
    SelectState* sel = reinterpret_cast<SelectState*>(hist + 3 * kHistBins);
    uint32_t* keys = reinterpret_cast<uint32_t*>(ws + ext_keys_off(N));
    const unsigned grid = static_cast<unsigned>(blocks);
    // the histogram passes: as many blocks as fit on the SMs, striding over the slices
    const size_t smem0 = hist_smem_bytes<0>(), smem12 = hist_smem_bytes<1>();
    const size_t per_sm0 = std::min<size_t>(kHistBlocksPerSm, (200u << 10) / smem0);
    const unsigned hgrid0 =
        static_cast<unsigned>(std::min<size_t>(blocks, static_cast<size_t>(sms) * per_sm0));
    const unsigned hgrid =
        static_cast<unsigned>(std::min<size_t>(blocks, static_cast<size_t>(sms) * kHistBlocksPerSm));
    const int64_t slices = static_cast<int64_t>(blocks);
    if (blocks > 0) {
        cudaError_t e = cudaFuncSetAttribute(audit_ext_hist<0>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem0));
        if (e != cudaSuccess) return e;
    }
    if (blocks > 0) {
        if (vec_ok)
            audit_ext_pass1<true><<<grid, kAuditThreads, 0, stream>>>(logp_new, logp_old, mask, N,
                                                                      eps, parts, keys);
        else
            audit_ext_pass1<false><<<grid, kAuditThreads, 0, stream>>>(logp_new, logp_old, mask,
                                                                       N, eps, parts, keys);
    }
    audit_ext_merge<<<1, kMergeThreads, 0, stream>>>(parts, static_cast<int64_t>(blocks),
                                                     seq_offsets, num_seqs, result, sel, hist);
    if (blocks > 0) {
        audit_ext_hist<0><<<hgrid0, kAuditThreads, smem0, stream>>>(keys, N, slices, sel, hist);
        audit_ext_select<0><<<1, kSelectThreads, 0, stream>>>(sel, hist, result);
        audit_ext_hist<1><<<hgrid, kAuditThreads, smem12, stream>>>(keys, N, slices, sel, hist);
        audit_ext_select<1><<<1, kSelectThreads, 0, stream>>>(sel, hist, result);
        audit_ext_hist<2><<<hgrid, kAuditThreads, smem12, stream>>>(keys, N, slices, sel, hist);
        audit_ext_select<2><<<1, kSelectThreads, 0, stream>>>(sel, hist, result);
    }
    return cudaGetLastError();
}

}  // namespace rlk
