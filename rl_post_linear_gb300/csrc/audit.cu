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

// Per-thread state of one slice: the active count, the slice's largest |d| as an
// order-preserving integer key (0: no active element) and the offset of its first
// occurrence (set only when it beats the thread's running best), and fp32 sums.
struct ThreadAcc {
    int count = 0;
    uint32_t key = 0;
    int arg = -1;
    float sd = 0.f, skl = 0.f;
    uint32_t flags = 0;
};

// The extended audit's terms of one slice seen by one thread: the sum of |d| and
// the count of clipped ratios (outputs); where the slice's keys go, the block's
// coarse histogram, the count of exact zeros and the clip thresholds (inputs).
struct ExtSlice {
    float sabs = 0.f;
    int clip = 0;
    uint32_t* keys;        // the slice's keys in global memory (element 0 of the slice)
    int64_t valid;         // elements of the slice inside N
    uint32_t* hist;        // coarse histogram in shared memory
    uint32_t n_zero;       // running count of |d| == 0 (kept in a register)
    float clip_lo, clip_hi;
};

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

constexpr int kCoarseWindowLo = 96;                   // exponent field of 2^-31
constexpr int kCoarseOctaves = 32;                    // window [2^-31, 2)
constexpr int kCoarseSub = 128;                       // bins per octave (7 mantissa bits)
constexpr int kCoarseZero = 0;                        // |d| == 0
constexpr int kCoarseLow = 1;                         // 0 < |d| < 2^-31
constexpr int kCoarseFirst = 2;                       // first bin of the window
constexpr int kCoarseHigh = kCoarseFirst + kCoarseOctaves * kCoarseSub;   // |d| >= 2, inf, NaN
constexpr int kCoarseBins = kCoarseHigh + 1;          // 4099

// bin = (b >> 16) - kCoarseShift inside the window (b = the |d| bits)
constexpr int kCoarseShift = (kCoarseWindowLo << 7) - kCoarseFirst;     // 12286
static_assert(kCoarseSub == 128, "bits 30..16 address the window's bins");

// The keys of coarse bin `bin` are the range [lo, lo + span) (the bins preserve order).
__device__ __forceinline__ void coarse_bin_keys(int bin, uint32_t& lo, uint32_t& span) {
    if (bin == kCoarseZero) {
        lo = 1u;
        span = 1u;
    } else if (bin == kCoarseLow) {
        lo = 2u;
        span = (static_cast<uint32_t>(kCoarseWindowLo) << 23) - 1u;
    } else if (bin == kCoarseHigh) {
        lo = (static_cast<uint32_t>(kCoarseWindowLo + kCoarseOctaves) << 23) + 1u;
        span = 0x7fc00001u - lo + 1u;
    } else {
        lo = (static_cast<uint32_t>(bin + kCoarseShift) << 16) + 1u;
        span = 0x10000u;
    }
}

// Coarse bin of nonzero |d| bits b (the key minus 1).  Bits 30..16 of b are the
// exponent and the top 7 mantissa bits, so inside the window the bin is
// (b >> 16) - (96 << 7) + kCoarseFirst; below and above the window the same value
// clamps to kCoarseLow and kCoarseHigh (any NaN lands there too); b = 0 is
// kCoarseZero, counted apart.
__device__ __forceinline__ int coarse_bin_nonzero(uint32_t bits) {
    return min(max(static_cast<int>(bits >> 16) - kCoarseShift, kCoarseLow), kCoarseHigh);
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
template <bool EXT = false>
__device__ __forceinline__ void visit_slice(const float4 (&x)[kVec], const float4 (&y)[kVec],
                                            const uint32_t (&m)[kVec], int tid, uint32_t best_key,
                                            ThreadAcc& a, ExtSlice* ext = nullptr) {
    float sd[kVec], skl[kVec], sab[kVec];
    uint32_t gmax[kVec];
    int clip = 0;
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        a.count += active_bytes(m[j]);
        const float xs[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
        const float ys[4] = {y[j].x, y[j].y, y[j].z, y[j].w};
        sd[j] = 0.f;
        skl[j] = 0.f;
        sab[j] = 0.f;
        gmax[j] = 0u;
        uint32_t k4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const bool act = ((m[j] >> (8 * e)) & 0xffu) != 0u;
            const float d = act ? xs[e] - ys[e] : 0.f;
            const uint32_t bits = __float_as_uint(d) & 0x7fffffffu;
            gmax[j] = max(gmax[j], bits);
            sd[j] += d;
            skl[j] += kl_small(d);
            if constexpr (EXT) {
                // |exp(d) - 1| > eps  <=>  d > log1p(eps) or d < log1p(-eps); d = 0 when inactive
                sab[j] += __uint_as_float(bits);
                clip += (d > ext->clip_hi || d < ext->clip_lo) ? 1 : 0;
                k4[e] = act ? key_of_bits(bits) : 0u;
                ext->n_zero += (act && bits == 0u) ? 1u : 0u;
                if (act && bits != 0u) atomicAdd(&ext->hist[coarse_bin_nonzero(bits)], 1u);
            }
        }
        if constexpr (EXT) {          // the group's keys (0 for inactive elements)
            const int o = j * (kAuditThreads * 4) + tid * 4;
            if (o + 4 <= ext->valid) {
                *reinterpret_cast<uint4*>(ext->keys + o) = make_uint4(k4[0], k4[1], k4[2], k4[3]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (o + e < ext->valid) ext->keys[o + e] = k4[e];
            }
        }
    }
    if constexpr (EXT) {
        ext->sabs = (sab[0] + sab[1]) + (sab[2] + sab[3]);
        ext->clip = clip;
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
template <bool VEC, bool EXT = false>
__device__ __forceinline__ void load_and_visit_slice(const float* nw, const float* od,
                                                     const uint8_t* mask, int64_t N,
                                                     int64_t base, uint32_t best_key,
                                                     ThreadAcc& a, ExtSlice* ext = nullptr) {
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
    visit_slice<EXT>(x, y, m, threadIdx.x, best_key, a, ext);
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
// partials in warp order, returned in thread 0 (unspecified in the others).
__device__ __forceinline__ AuditPartial block_partial(RunAcc r) {
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
    AuditPartial p{};
    if (threadIdx.x == 0) {
        Acc t = warp_acc[0];
#pragma unroll
        for (int w = 1; w < kAuditThreads / 32; ++w) merge(t, warp_acc[w]);
        p.count = t.count;
        p.arg = t.arg;
        p.sum_d = t.sum_d;
        p.sum_kl = t.sum_kl;
        p.best = t.best;
        p.flags = t.flags;
    }
    return p;
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
    const AuditPartial p = block_partial(r);
    if (threadIdx.x == 0) out[blockIdx.x] = p;
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
// position.
//
//   pass 1   the base audit's slices and blocks, plus per thread the sum of |d|
//            and the clip count; it writes each element's |d| key (the order-
//            preserving key of the base audit, 0 for inactive elements) and
//            counts the keys into a coarse histogram: exact zeros, keys below
//            2^-31, 128 bins per octave over [2^-31, 2), keys from 2 up (inf
//            and NaN included) -- per block in shared memory, then added to a
//            global one with integer atomics.
//   merge    one block: the fixed-order merge of the partials, and for each
//            percentile the coarse bin holding its rank, with the number of
//            keys below that bin (an exact integer).
//   pass 2   reads the keys once and appends those in each percentile's bin to
//            that percentile's candidate list (in any order: only the multiset
//            matters).
//   select   an exact radix select of the remaining rank among each list's
//            keys (two 8-bit digits inside a bin of the window, three digits of
//            11, 11 and 9 bits in the bins outside it), counted with integer
//            histograms.
// Mean ratio0 = 1 + mean(d) + mean(exp(d) - 1 - d), from the sums the base audit
// already forms (exact algebra; no exp per element).  The clip test
// |exp(d) - 1| > eps is d > log1p(eps) or d < log1p(-eps), the two thresholds
// rounded to fp32 on the host.  Every count is an integer, so the selected
// values, like the sums, are bitwise reproducible for a given N.

struct ExtPartial {
    AuditPartial base;
    DFloat sum_abs;
    int64_t clip;
};

constexpr int kSelBins = 2048;
constexpr int kSelPasses = 3;

// The selection of one percentile after some radix passes.
struct SelState {
    int64_t rank;          // 1-based rank left to select among the matching keys; 0: none
    uint32_t kmask;        // bits of the |d| bits already fixed ...
    uint32_t kvalue;       // ... and their values
    int32_t done;          // 1: the value is kvalue
    int32_t pad;
};

// The selection state of the three percentiles (p50, p90, p99).  st[p] is the
// state before radix pass p (st[0] from the merge); the kernel of pass p writes
// st[p] from st[p - 1], so no kernel overwrites what its own blocks read.
struct ExtSelect {
    unsigned long long cand_count[3];   // candidates appended by pass 2
    int32_t bin[3];                     // coarse bin of the rank
    int32_t pad;
    SelState st[kSelPasses][3];
};

// the radix digit of pass p for a percentile in coarse bin `bin` (bits == 0: no pass)
__device__ __forceinline__ void sel_digit(int bin, int p, int& shift, int& bits) {
    if (bin >= kCoarseFirst && bin < kCoarseHigh) {     // the low 16 bits vary inside a bin
        shift = p == 0 ? 8 : 0;
        bits = p < 2 ? 8 : 0;
    } else {                                              // all 31 bits vary
        shift = p == 0 ? 20 : (p == 1 ? 9 : 0);
        bits = p < 2 ? 11 : 9;
    }
}

// The extended pass 1 deals the slices to min(slices, kExtMaxBlocks) blocks (a fixed
// partition of its own: three of its blocks are resident on each of 152 SMs).
constexpr int64_t kExtMaxBlocks = 456;

template <bool VEC>
__global__ void __launch_bounds__(kAuditThreads, 3)
    audit_ext_pass1(const float* __restrict__ nw, const float* __restrict__ od,
                    const uint8_t* __restrict__ mask, int64_t N, float clip_lo, float clip_hi,
                    ExtPartial* __restrict__ out, uint32_t* __restrict__ keys,
                    unsigned long long* __restrict__ coarse) {
    __shared__ uint32_t h[kCoarseBins];
    for (int i = threadIdx.x; i < kCoarseBins; i += kAuditThreads) h[i] = 0u;
    __syncthreads();
    const int64_t slices = (N + kSlice - 1) / kSlice;
    RunAcc r;
    DFloat sabs{0.f, 0.f};
    int clip = 0;
    ExtSlice x;
    x.hist = h;
    x.n_zero = 0u;
    x.clip_lo = clip_lo;
    x.clip_hi = clip_hi;
#pragma unroll 1
    for (int64_t sl = blockIdx.x; sl < slices; sl += gridDim.x) {
        const int64_t base = sl * kSlice;
        ThreadAcc a;
        x.keys = keys + base;
        x.valid = N - base;
        load_and_visit_slice<VEC, true>(nw, od, mask, N, base, r.best_key, a, &x);
        r.add_slice(a, base);
        sabs = df_add(sabs, DFloat{x.sabs, 0.f});
        clip += x.clip;
    }
    uint32_t n_zero = x.n_zero;
    // the block's partial: the base audit's tree, then the same tree for |d| and the clips
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        DFloat y;
        y.hi = __shfl_down_sync(0xffffffffu, sabs.hi, off);
        y.lo = __shfl_down_sync(0xffffffffu, sabs.lo, off);
        const int c = __shfl_down_sync(0xffffffffu, clip, off);
        const uint32_t z0 = __shfl_down_sync(0xffffffffu, n_zero, off);
        if (lane + off < 32) {
            sabs = df_add(sabs, y);
            clip += c;
            n_zero += z0;
        }
    }
    __shared__ DFloat w_abs[kAuditThreads / 32];
    __shared__ int w_clip[kAuditThreads / 32];
    if (lane == 0) {
        w_abs[warp] = sabs;
        w_clip[warp] = clip;
        if (n_zero) atomicAdd(&h[kCoarseZero], n_zero);
    }
    const AuditPartial bp = block_partial(r);      // its barrier also orders the writes above
    for (int i = threadIdx.x; i < kCoarseBins; i += kAuditThreads)
        if (h[i] != 0u) atomicAdd(&coarse[i], static_cast<unsigned long long>(h[i]));
    if (threadIdx.x == 0) {
        DFloat sa = w_abs[0];
        int64_t cl = w_clip[0];
#pragma unroll
        for (int w = 1; w < kAuditThreads / 32; ++w) {
            sa = df_add(sa, w_abs[w]);
            cl += w_clip[w];
        }
        ExtPartial ep;
        ep.base = bp;
        ep.sum_abs = sa;
        ep.clip = cl;
        out[blockIdx.x] = ep;
    }
}

// One block: the fixed-order merge of the partials; writes the sums into the
// result; for each percentile the coarse bin holding its rank and the rank left
// inside it; clears the candidate counts and the select histograms.
__global__ void __launch_bounds__(kMergeThreads)
    audit_ext_merge(const ExtPartial* __restrict__ parts, int64_t num_parts,
                    const int64_t* __restrict__ seq_offsets, int64_t num_seqs,
                    const unsigned long long* __restrict__ coarse,
                    rlk_audit_ext_t* __restrict__ result, ExtSelect* __restrict__ sel,
                    unsigned long long* __restrict__ sel_hist) {
    Acc a = empty_acc();
    DFloat sa{0.f, 0.f};
    int64_t cl = 0;
    // ascending partials per thread, loaded in batches (as in the base audit's merge)
    auto fold = [&](const ExtPartial& p) {
        merge(a, to_acc(p.base));
        sa = df_add(sa, p.sum_abs);
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
    for (int k = threadIdx.x; k < kSelPasses * 3 * kSelBins; k += kMergeThreads) sel_hist[k] = 0ull;
    a = block_reduce<kMergeThreads>(a);
    __shared__ DFloat s_abs[kMergeThreads / 32];
    __shared__ long long s_clip[kMergeThreads / 32];
    __shared__ long long s_count;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // the same fixed tree for the two extra sums
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        DFloat x;
        x.hi = __shfl_down_sync(0xffffffffu, sa.hi, off);
        x.lo = __shfl_down_sync(0xffffffffu, sa.lo, off);
        const long long z = __shfl_down_sync(0xffffffffu, static_cast<long long>(cl), off);
        if (lane + off < 32) {
            sa = df_add(sa, x);
            cl += z;
        }
    }
    if (lane == 0) {
        s_abs[warp] = sa;
        s_clip[warp] = cl;
    }
    if (threadIdx.x == 0) s_count = a.count;
    __syncthreads();
    const int64_t count = s_count;
    if (threadIdx.x == 0) {
        for (int w = 1; w < kMergeThreads / 32; ++w) {
            s_abs[0] = df_add(s_abs[0], s_abs[w]);
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
        r.approx_kl = df_value(a.sum_kl) / cnt;
        // mean exp(d) = 1 + mean d + mean (exp(d) - 1 - d)
        r.mean_ratio = (cnt + df_value(a.sum_d) + df_value(a.sum_kl)) / cnt;
        r.max_abs_dlogp = a.count > 0 ? a.best : 0.0f;
        r.p50_abs_dlogp = r.p90_abs_dlogp = r.p99_abs_dlogp = __int_as_float(0x7fc00000);
        r.clipfrac = static_cast<float>(static_cast<double>(s_clip[0]) / cnt);
        r.error_flags = a.flags;
        *result = r;
    }
    // each percentile's coarse bin: an exclusive scan of the bins (integers, so exact),
    // five consecutive bins per thread; the one thread whose run holds the rank walks it
    constexpr int kRun = (kCoarseBins + kMergeThreads - 1) / kMergeThreads;   // 5
    __shared__ unsigned long long warp_sum[kMergeThreads / 32];
    // defaults (no active token: done, rank 0), overwritten below by the thread that finds
    // each rank; the barrier of the scan orders the two
    if (threadIdx.x < 3) {
        SelState st;
        st.rank = 0;
        st.kmask = 0u;
        st.kvalue = 0u;
        st.done = 1;
        st.pad = 0;
        sel->cand_count[threadIdx.x] = 0ull;
        sel->bin[threadIdx.x] = -1;
        sel->st[0][threadIdx.x] = st;
    }
    unsigned long long c[kRun];
    unsigned long long run = 0;
#pragma unroll
    for (int j = 0; j < kRun; ++j) {
        const int b = threadIdx.x * kRun + j;
        c[j] = b < kCoarseBins ? coarse[b] : 0ull;
        run += c[j];
    }
    unsigned long long incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    unsigned long long before = 0;
    for (int w = 0; w < warp; ++w) before += warp_sum[w];
    const unsigned long long excl = before + incl - run;
    const int pct[3] = {50, 90, 99};
    for (int q = 0; q < 3; ++q) {
        const int64_t rank = (pct[q] * count + 99) / 100;   // nearest rank, 1-based (0 if none)
        if (rank <= 0) continue;                            // st[0][q] says done, rank 0
        const unsigned long long rk = static_cast<unsigned long long>(rank);
        if (excl < rk && rk <= excl + run) {               // exactly one thread
            unsigned long long cum = excl;
            int bin = -1;
#pragma unroll
            for (int j = 0; j < kRun; ++j) {
                if (bin < 0) {
                    if (rk <= cum + c[j]) bin = threadIdx.x * kRun + j;
                    else cum += c[j];
                }
            }
            SelState st;
            st.rank = static_cast<int64_t>(rk - cum);
            st.kmask = 0u;
            st.kvalue = 0u;
            st.done = 0;
            st.pad = 0;
            if (bin == kCoarseZero) {                 // every key in the bin is |d| = 0
                st.done = 1;
            } else if (bin >= kCoarseFirst && bin < kCoarseHigh) {
                // the bin fixes the exponent and the top 7 mantissa bits
                st.kmask = 0x7fff0000u;
                st.kvalue =
                    (static_cast<uint32_t>((bin - kCoarseFirst) >> 7) + kCoarseWindowLo) << 23 |
                    (static_cast<uint32_t>((bin - kCoarseFirst) & 0x7f) << 16);
            }
            sel->bin[q] = bin;
            sel->st[0][q] = st;
        }
    }
}

// Pass 2 puts every key in a percentile's coarse bin in that percentile's candidate
// list, in any order (only the multiset matters); kCandStage keys per list are
// staged in shared memory first.
constexpr int kCandStage = 2048;

__device__ __forceinline__ void collect_key(uint32_t key, const uint32_t (&lo)[3],
                                            const uint32_t (&span)[3], unsigned* s_n,
                                            uint32_t (*stage)[kCandStage], ExtSelect* sel,
                                            uint32_t* cand, int64_t cand_stride) {
#pragma unroll
    for (int q = 0; q < 3; ++q) {
        if (key - lo[q] < span[q]) {          // inactive keys (0) are below every range
            const unsigned pos = atomicAdd(&s_n[q], 1u);
            if (pos < kCandStage) {
                stage[q][pos] = key;
            } else {                  // the stage is full: straight to the global list
                const unsigned long long g = atomicAdd(&sel->cand_count[q], 1ull);
                cand[q * cand_stride + static_cast<int64_t>(g)] = key;
            }
        }
    }
}

// Pass 2 reads the keys as a plain stream (16 bytes per thread and iteration, the
// whole grid sweeping them front to back; the candidate multiset does not depend on
// it).  A block stages its candidates in shared memory (a shared atomic per
// candidate: they are rare) and, at the end, reserves room in each global list with
// one atomic; what does not fit in the stage goes to the global list at once.
__global__ void __launch_bounds__(kAuditThreads)
    audit_ext_collect(const uint32_t* __restrict__ keys, int64_t N, ExtSelect* __restrict__ sel,
                      uint32_t* __restrict__ cand, int64_t cand_stride) {
    __shared__ uint32_t stage[3][kCandStage];
    __shared__ unsigned s_n[3];
    __shared__ unsigned long long s_base[3];
    // each percentile's key range; an empty range (span 0) for one already known
    uint32_t lo[3], span[3];
    bool need = false;
#pragma unroll
    for (int q = 0; q < 3; ++q) {
        lo[q] = 0u;
        span[q] = 0u;
        if (!sel->st[0][q].done) {
            coarse_bin_keys(sel->bin[q], lo[q], span[q]);
            need = true;
        }
    }
    if (!need) return;
    if (threadIdx.x < 3) s_n[threadIdx.x] = 0u;
    __syncthreads();
    const int64_t n4 = N / 4;
    const uint4* k4 = reinterpret_cast<const uint4*>(keys);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kAuditThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kAuditThreads + threadIdx.x; i < n4;
         i += stride) {
        const uint4 v = __ldcs(k4 + i);
        collect_key(v.x, lo, span, s_n, stage, sel, cand, cand_stride);
        collect_key(v.y, lo, span, s_n, stage, sel, cand, cand_stride);
        collect_key(v.z, lo, span, s_n, stage, sel, cand, cand_stride);
        collect_key(v.w, lo, span, s_n, stage, sel, cand, cand_stride);
    }
    if (blockIdx.x == 0 && threadIdx.x < N - n4 * 4)     // the last N mod 4 keys
        collect_key(keys[n4 * 4 + threadIdx.x], lo, span, s_n, stage, sel, cand, cand_stride);
    __syncthreads();
    if (threadIdx.x < 3) {
        const unsigned n = min(s_n[threadIdx.x], static_cast<unsigned>(kCandStage));
        s_base[threadIdx.x] = n > 0u ? atomicAdd(&sel->cand_count[threadIdx.x],
                                                 static_cast<unsigned long long>(n))
                                     : 0ull;
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 3; ++q) {
        const unsigned n = min(s_n[q], static_cast<unsigned>(kCandStage));
        for (unsigned i = threadIdx.x; i < n; i += kAuditThreads)
            cand[q * cand_stride + static_cast<int64_t>(s_base[q]) + i] = stage[q][i];
    }
}

// The select step after radix pass p of percentile q: the digit whose bin holds
// the rank (an exclusive scan of the 2^bits counts, exact), appended to the known
// bits.  Run identically by every block of the next pass and by the final step.
__device__ void sel_step(int q, int p, int bin, const unsigned long long* __restrict__ sel_hist,
                         SelState& st) {
    __shared__ unsigned long long warp_sum[kAuditThreads / 32];
    __shared__ uint32_t s_digit;
    __shared__ int64_t s_rank;
    int shift, bits;
    sel_digit(bin, p, shift, bits);
    if (st.done || bits == 0) return;                  // block-uniform
    if (threadIdx.x == 0) {                            // (always overwritten: the counts are exact)
        s_digit = 0u;
        s_rank = 1;
    }
    const int nb = 1 << bits;
    const int runl = nb / kAuditThreads;                 // 8, or 2 for 9 bits
    const unsigned long long* hq = sel_hist + (static_cast<int64_t>(p) * 3 + q) * kSelBins;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long c[8];
    unsigned long long run = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        c[j] = j < runl ? hq[threadIdx.x * runl + j] : 0ull;
        run += c[j];
    }
    unsigned long long incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    unsigned long long before = 0;
    for (int w = 0; w < warp; ++w) before += warp_sum[w];
    const unsigned long long excl = before + incl - run;
    const unsigned long long rk = static_cast<unsigned long long>(st.rank);
    if (excl < rk && rk <= excl + run) {
        unsigned long long cum = excl;
        int dg = -1;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (dg < 0 && j < runl) {
                if (rk <= cum + c[j]) dg = threadIdx.x * runl + j;
                else cum += c[j];
            }
        }
        s_digit = static_cast<uint32_t>(dg);
        s_rank = static_cast<int64_t>(rk - cum);
    }
    __syncthreads();
    const uint32_t dmask = static_cast<uint32_t>(nb - 1) << shift;
    st.kmask |= dmask;
    st.kvalue = (st.kvalue & ~dmask) | (s_digit << shift);
    st.rank = s_rank;
    int s2, b2;
    sel_digit(bin, p + 1, s2, b2);
    st.done = (p + 1 >= kSelPasses || b2 == 0) ? 1 : 0;
    __syncthreads();
}

// Radix pass p over each percentile's candidates (blockIdx.y = percentile): the
// histogram of digit p among the candidates that match the bits known so far.
// For p > 0 every block first repeats the select step of pass p - 1; block 0
// stores its outcome.
template <int P>
__global__ void __launch_bounds__(kAuditThreads)
    audit_ext_radix(ExtSelect* __restrict__ sel, const uint32_t* __restrict__ cand,
                    int64_t cand_stride, unsigned long long* __restrict__ sel_hist) {
    const int q = blockIdx.y;
    const int bin = sel->bin[q];
    SelState st = sel->st[P == 0 ? 0 : P - 1][q];
    if (P > 0) {
        sel_step(q, P - 1, bin, sel_hist, st);
        if (blockIdx.x == 0 && threadIdx.x == 0) sel->st[P][q] = st;
    }
    if (st.done) return;                                // block-uniform
    const uint32_t kmask = st.kmask, kvalue = st.kvalue;
    int shift, bits;
    sel_digit(bin, P, shift, bits);
    const uint32_t dmask = (1u << bits) - 1u;
    __shared__ uint32_t h[kSelBins];
    for (int i = threadIdx.x; i < kSelBins; i += kAuditThreads) h[i] = 0u;
    __syncthreads();
    const int64_t n = static_cast<int64_t>(sel->cand_count[q]);
    const uint32_t* cq = cand + q * cand_stride;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kAuditThreads + threadIdx.x; i - threadIdx.x < n;
         i += static_cast<int64_t>(gridDim.x) * kAuditThreads) {
        const bool in = i < n;
        const uint32_t b = in ? cq[i] - 1u : 0u;
        const bool match = in && (b & kmask) == kvalue;
        const uint32_t digit = (b >> shift) & dmask;
        // equal digits within the warp add up in one atomic (many equal keys are common)
        const unsigned act = __ballot_sync(0xffffffffu, match);
        if (match) {
            const unsigned peers = __match_any_sync(act, digit);
            if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&h[digit], __popc(peers));
        }
    }
    __syncthreads();
    unsigned long long* gh = sel_hist + (static_cast<int64_t>(P) * 3 + q) * kSelBins;
    for (int i = threadIdx.x; i < (1 << bits); i += kAuditThreads)
        if (h[i] != 0u) atomicAdd(&gh[i], static_cast<unsigned long long>(h[i]));
}

// The last select step; the selected |d| bits become p50 / p90 / p99.
__global__ void __launch_bounds__(kAuditThreads)
    audit_ext_finish(const ExtSelect* __restrict__ sel,
                     const unsigned long long* __restrict__ sel_hist,
                     rlk_audit_ext_t* __restrict__ result) {
    for (int q = 0; q < 3; ++q) {
        SelState st = sel->st[kSelPasses - 1][q];
        if (st.rank <= 0) continue;                      // no active token: NaN stays
        sel_step(q, kSelPasses - 1, sel->bin[q], sel_hist, st);
        if (threadIdx.x == 0) {
            const float v = __uint_as_float(st.kvalue);
            if (q == 0) result->p50_abs_dlogp = v;
            if (q == 1) result->p90_abs_dlogp = v;
            if (q == 2) result->p99_abs_dlogp = v;
        }
    }
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

// extended audit workspace: partials | coarse histogram | select state | select
// histograms | |d| keys [N] | candidate lists [3][N] (uint32)
struct ExtLayout {
    size_t coarse_off, sel_off, hist_off, keys_off, cand_off, total;
    explicit ExtLayout(int64_t N) {
        coarse_off = align_up(static_cast<size_t>(kExtMaxBlocks) * sizeof(ExtPartial), 256);
        sel_off = align_up(coarse_off + kCoarseBins * sizeof(unsigned long long), 256);
        hist_off = align_up(sel_off + sizeof(ExtSelect), 256);
        keys_off = align_up(hist_off + kSelPasses * 3 * kSelBins * sizeof(unsigned long long), 256);
        cand_off = align_up(keys_off + static_cast<size_t>(N) * 4, 256);
        total = align_up(cand_off + 3 * static_cast<size_t>(N) * 4, 256) + 256;
    }
};

size_t audit_ext_workspace(int64_t N) { return ExtLayout(N).total; }

cudaError_t launch_audit_ext(const float* logp_new, const float* logp_old, const uint8_t* mask,
                             int64_t N, const int64_t* seq_offsets, int64_t num_seqs, float eps,
                             rlk_audit_ext_t* result, void* workspace, bool vec_ok, int sms,
                             cudaStream_t stream) {
    const ExtLayout lay(N);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    ExtPartial* parts = reinterpret_cast<ExtPartial*>(ws);
    unsigned long long* coarse = reinterpret_cast<unsigned long long*>(ws + lay.coarse_off);
    ExtSelect* sel = reinterpret_cast<ExtSelect*>(ws + lay.sel_off);
    unsigned long long* sel_hist = reinterpret_cast<unsigned long long*>(ws + lay.hist_off);
    uint32_t* keys = reinterpret_cast<uint32_t*>(ws + lay.keys_off);
    uint32_t* cand = reinterpret_cast<uint32_t*>(ws + lay.cand_off);
    const int64_t cand_stride = N;
    // the clip thresholds of |exp(d) - 1| > eps, rounded to fp32 once
    const double e = static_cast<double>(eps);
    const float clip_hi = static_cast<float>(std::log1p(e));
    const float clip_lo = e < 1.0 ? static_cast<float>(std::log1p(-e)) : -INFINITY;
    const int64_t slices = static_cast<int64_t>(audit_v3_blocks(N));
    const unsigned blocks = static_cast<unsigned>(std::min<int64_t>(slices, kExtMaxBlocks));
    cudaError_t err = cudaMemsetAsync(coarse, 0, kCoarseBins * sizeof(unsigned long long), stream);
    if (err != cudaSuccess) return err;
    if (blocks > 0) {
        if (vec_ok)
            audit_ext_pass1<true><<<blocks, kAuditThreads, 0, stream>>>(
                logp_new, logp_old, mask, N, clip_lo, clip_hi, parts, keys, coarse);
        else
            audit_ext_pass1<false><<<blocks, kAuditThreads, 0, stream>>>(
                logp_new, logp_old, mask, N, clip_lo, clip_hi, parts, keys, coarse);
    }
    audit_ext_merge<<<1, kMergeThreads, 0, stream>>>(parts, static_cast<int64_t>(blocks),
                                                     seq_offsets, num_seqs, coarse, result, sel,
                                                     sel_hist);
    if (blocks > 0) {
        // the candidate scan: eight blocks per SM at most (the candidate lists do not depend
        // on the grid)
        const unsigned cgrid = static_cast<unsigned>(std::max<int64_t>(
            1, std::min<int64_t>((N / 4 + kAuditThreads - 1) / kAuditThreads,
                                 8 * static_cast<int64_t>(sms > 0 ? sms : 1))));
        audit_ext_collect<<<cgrid, kAuditThreads, 0, stream>>>(keys, N, sel, cand, cand_stride);
        const dim3 rg(blocks, 3);
        audit_ext_radix<0><<<rg, kAuditThreads, 0, stream>>>(sel, cand, cand_stride, sel_hist);
        audit_ext_radix<1><<<rg, kAuditThreads, 0, stream>>>(sel, cand, cand_stride, sel_hist);
        audit_ext_radix<2><<<rg, kAuditThreads, 0, stream>>>(sel, cand, cand_stride, sel_hist);
        audit_ext_finish<<<1, kAuditThreads, 0, stream>>>(sel, sel_hist, result);
    }
    return cudaGetLastError();
}

}  // namespace rlk
