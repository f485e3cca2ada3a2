// audit.cu -- deterministic masked dlogp audit.
//
// "RL-Kernel integration roadmap for vime", Consistency Contract:
// dlogp = recomputed - old; every aggregate over active tokens only;
// max_abs_dlogp is the primary metric, reported with the worst token;
// approx_kl0 = mean(exp(dlogp) - 1 - dlogp); the active-token count.
//
// Pass 1: the elements are cut into 4096-element slices, dealt round-robin to
// G = min(slices, 608) blocks (block b takes slices b, b + G, b + 2G, ...: a
// function of N only, so that one wave of blocks covers any N and the grid
// sweeps the inputs front to back together).  For each slice a thread
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
#include <cstddef>
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

// a - b as the 64-bit multiply-add a * one + (2^64 - b) (one = 1): the high word is
// all ones exactly when a < b (unsigned), the low word is a - b mod 2^32.  (This
// form of the window tests below measured faster than compares and selects.)
__device__ __forceinline__ uint64_t sub_wide(uint32_t a, uint64_t neg_b, uint32_t one) {
    uint64_t t;
    asm("mad.wide.u32 %0, %1, %2, %3;" : "=l"(t) : "r"(a), "r"(one), "l"(neg_b));
    return t;
}

// acc + m * k (low 32 bits)
__device__ __forceinline__ uint32_t mad_lo(uint32_t m, uint32_t k, uint32_t acc) {
    uint32_t r;
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(r) : "r"(m), "r"(k), "r"(acc));
    return r;
}

// The extended audit's terms of one slice seen by one thread: the sum of |d| and
// the count of clipped ratios (outputs, per slice); per percentile q the count of
// active keys below its window (running over the thread's slices).  The keys inside
// window q are appended to the warp's own range of list q: `cand` + q * `qstride`,
// `n[q]` keys so far (the same value in every lane).  Given: the windows
// [lo, lo + span] of keys and the clip thresholds.
struct ExtSlice {
    float sabs = 0.f;
    int clip = 0;
    uint32_t below[3] = {0u, 0u, 0u};     // keys below window q, inactive elements included
    uint32_t n[3] = {0u, 0u, 0u};
    uint32_t lo[3], span[3];
    uint64_t neg_lo[3], neg_size[3];      // 2^64 - lo, 2^64 - (span + 1)
    uint32_t one, neg_one;                // 1 and 2^32 - 1
    float clip_lo, clip_hi;
    uint32_t* cand;
    int64_t qstride;
    uint32_t (*skeys)[kAuditThreads];     // [16][threads] in shared memory: the slice's keys
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
    uint32_t inw[3] = {0u, 0u, 0u};       // EXT: elements inside each window (bit 4j + e)
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        a.count += active_bytes(m[j]);
        const float xs[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
        const float ys[4] = {y[j].x, y[j].y, y[j].z, y[j].w};
        sd[j] = 0.f;
        skl[j] = 0.f;
        sab[j] = 0.f;
        gmax[j] = 0u;
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
                // the key (0 when inactive); u = key - lo wraps, so that an active key is
                // below window q exactly when u > -lo (key 0 gives u = -lo: never) and
                // inside it when u <= span.  Elements inside a window are marked (bit 4j + e) and their
                // keys listed after the loop.
                const uint32_t key = act ? key_of_bits(bits) : 0u;
                ext->skeys[4 * j + e][tid] = key;
#pragma unroll
                for (int q = 0; q < 3; ++q) {
                    // below: key < lo (key 0 too: the inactive are taken off per slice);
                    // inside: key - lo < span + 1 (key 0 wraps far above)
                    const uint64_t t = sub_wide(key, ext->neg_lo[q], ext->one);
                    ext->below[q] = mad_lo(static_cast<uint32_t>(t >> 32), ext->neg_one, ext->below[q]);
                    const uint64_t v = sub_wide(static_cast<uint32_t>(t), ext->neg_size[q], ext->one);
                    inw[q] = mad_lo(static_cast<uint32_t>(v >> 32), 0u - (1u << (4 * j + e)), inw[q]);
                }
            }
        }
    }
    if constexpr (EXT) {
        // the warp's keys inside window q go to its range of list q in lane order
        const int lane = tid & 31;
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            if (__any_sync(0xffffffffu, inw[q] != 0u)) {            // warp-uniform
                const int c = __popc(inw[q]);
                int incl = c;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += v;
                }
                uint32_t* dst = ext->cand + q * ext->qstride + ext->n[q] + (incl - c);
                for (uint32_t m = inw[q]; m != 0u; m &= m - 1u) *dst++ = ext->skeys[__ffs(m) - 1][tid];
                ext->n[q] += static_cast<uint32_t>(__shfl_sync(0xffffffffu, incl, 31));
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
// inactive.  Either way the arithmetic that follows is the same.
template <bool VEC>
__device__ __forceinline__ void load_slice(const float* nw, const float* od, const uint8_t* mask,
                                           int64_t N, int64_t base, float4 (&x)[kVec],
                                           float4 (&y)[kVec], uint32_t (&m)[kVec],
                                           int tid = static_cast<int>(threadIdx.x)) {
    if (VEC && base + kSlice <= N) {
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const int64_t i0 = base + j * (kAuditThreads * 4) + tid * 4;
            x[j] = __ldcs(reinterpret_cast<const float4*>(nw + i0));
            y[j] = __ldcs(reinterpret_cast<const float4*>(od + i0));
            m[j] = mask == nullptr ? 0x01010101u
                                   : __ldcs(reinterpret_cast<const unsigned int*>(mask + i0));
        }
    } else {
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const int64_t i0 = base + j * (kAuditThreads * 4) + tid * 4;
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
}

template <bool VEC, bool EXT = false>
__device__ __forceinline__ void load_and_visit_slice(const float* nw, const float* od,
                                                     const uint8_t* mask, int64_t N,
                                                     int64_t base, uint32_t best_key,
                                                     ThreadAcc& a, ExtSlice* ext = nullptr) {
    float4 x[kVec], y[kVec];
    uint32_t m[kVec];
    load_slice<VEC>(nw, od, mask, N, base, x, y, m);
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
// position.  A percentile is an exact order statistic of the |d| keys (the
// base audit's order-preserving keys); it is found among a small candidate set
// that provably holds it, by an exact radix select with integer histograms.
//
//   sample   every K-th 4096-element slice (K a function of N: 128 to 255
//            slices in all, every slice of a smaller batch) is counted into a coarse histogram of |d|: exact
//            zeros, |d| below 2^-31, 128 bins per octave over [2^-31, 2), |d|
//            from 2 up (inf and NaN included).  The last block to finish
//            (an integer ticket) turns it into one window of keys per
//            percentile: the bins from sample rank r - w to r + w, where r is
//            the percentile's rank in the sample and w four standard
//            deviations of a sample rank plus 16.
//   main     the base audit's slices and blocks, plus per thread the sum of
//            |d|, the clip count, and per percentile the count of active keys
//            below its window; keys inside a window go to that percentile's
//            candidate list.
//   merge    one block: the fixed-order merge of the partials into the
//            result, and the check that each percentile's rank r falls inside
//            its window (below < r <= below + candidates, exact integers).
//   fallback only where the check failed (a sample that misrepresents the
//            whole, which the window makes improbable): an exact coarse
//            histogram of all keys, then the keys of the bin holding the rank
//            replace that percentile's candidates.  Launched always; it
//            returns at once when every check passed.
//   select   radix passes over the candidates that share the window's common
//            leading bits: digits of up to 11 bits, from the highest varying
//            bit down, each pass a histogram of the candidates that match the
//            digits chosen so far.
// The result never depends on the sample: it only decides how much work the
// selection takes.  Mean ratio0 = 1 + mean(d) + mean(exp(d) - 1 - d), from the
// sums the base audit already forms (exact algebra; no exp per element).  The
// clip test |exp(d) - 1| > eps is d > log1p(eps) or d < log1p(-eps), the two
// thresholds rounded to fp32 on the host.  Every count is an integer, so the
// selected values, like the sums, are bitwise reproducible for a given N.

struct ExtPartial {
    AuditPartial base;
    DFloat sum_abs;
    int64_t clip;
    int64_t below[3];
};

constexpr int kSelBins = 2048;
constexpr int kSelPasses = 3;
constexpr int kSelDigit = 11;          // bits of a radix digit

// percentile q of (p50, p90, p99)
__host__ __device__ __forceinline__ int pct_of(int q) { return q == 0 ? 50 : (q == 1 ? 90 : 99); }

// The selection of one percentile after some radix passes.
struct SelState {
    int64_t rank;          // 1-based rank left to select among the matching keys; 0: none
    uint32_t kmask;        // bits of the |d| bits already fixed ...
    uint32_t kvalue;       // ... and their values
    int32_t done;          // 1: the value is kvalue
    int32_t vbits;         // the low bits that vary inside the window
};

// The state shared by the extended audit's kernels.  st[p] is the state before
// radix pass p (st[0] from the merge or the fallback); the kernel of pass p
// writes st[p] from st[p - 1], so no kernel overwrites what its own blocks read.
struct ExtSelect {
    int64_t rank[3];                    // each percentile's rank among all active keys
    uint32_t win_lo[3];                 // each percentile's window of keys [lo, hi]
    uint32_t win_hi[3];
    int32_t fallback[3];                // 1: the window missed the rank
    int32_t need_fallback;
    SelState st[kSelPasses][3];
};

// Candidate lists.  The main pass (and the fallback, with the same blocks and
// slices) gives each warp a fixed range of every list, room for all the elements
// it visits: capw = 512 keys per slice of its block.  List q starts at q * qstride;
// the keys warp w of block b has put there are [(8 b + w) capw, + wn[q][8 b + w]).
constexpr int kWarps = kAuditThreads / 32;
constexpr int64_t kExtMaxBlocks = 456;             // three resident on each of 152 SMs
constexpr int64_t kWnStride = kExtMaxBlocks * kWarps;

struct ExtGeom {
    int64_t slices, blocks, capw, qstride;
    __host__ __device__ explicit ExtGeom(int64_t N) {
        slices = (N + kSlice - 1) / kSlice;
        blocks = slices < kExtMaxBlocks ? slices : kExtMaxBlocks;
        const int64_t per_block = blocks > 0 ? (slices + blocks - 1) / blocks : 0;
        capw = per_block * (kSlice / kWarps);
        qstride = blocks * kWarps * capw;
    }
};

// (The GPU tests read the fallback flags at this place in the workspace.)
static_assert(sizeof(ExtPartial) == 80 && offsetof(ExtSelect, fallback) == 48,
              "extended-audit workspace layout");

// The keys of coarse bin `bin` are the range [lo, hi] (the bins preserve order).
__device__ __forceinline__ void coarse_bin_range(int bin, uint32_t& lo, uint32_t& hi) {
    uint32_t span;
    coarse_bin_keys(bin, lo, span);
    hi = lo + span - 1u;
}

// The digit of radix pass p for a window whose low `vbits` bits vary (bits == 0: no pass).
__device__ __forceinline__ void sel_digit(int vbits, int p, int& shift, int& bits) {
    const int top = vbits - kSelDigit * p;
    shift = top > kSelDigit ? top - kSelDigit : 0;
    bits = top > 0 ? top - shift : 0;
}

// The state before the first radix pass for keys in [lo, hi] and the rank left
// among them: the common leading bits of the window are known.
__device__ __forceinline__ SelState window_state(uint32_t lo, uint32_t hi, int64_t rank) {
    const uint32_t a = lo - 1u, b = hi - 1u;          // |d| bits
    const uint32_t diff = a ^ b;
    SelState st;
    st.vbits = diff == 0u ? 0 : 32 - __clz(diff);
    st.kmask = st.vbits >= 32 ? 0u : (0xffffffffu << st.vbits);
    st.kvalue = a & st.kmask;
    st.rank = rank;
    st.done = st.vbits == 0 ? 1 : 0;
    return st;
}

// A coarse histogram held by the THREADS threads of a block, kRun consecutive bins
// each, with the exclusive prefix of each thread's run: find(r) locates the bin of
// 1-based rank r.  Loaded from u64 counts in global memory (through L2) or from
// u32 counts in shared memory.
template <int THREADS>
struct BinScan {
    static constexpr int kRun = (kCoarseBins + THREADS - 1) / THREADS;
    unsigned long long c[kRun];
    unsigned long long run, excl, total;

    __device__ void load(const unsigned long long* hist) {
#pragma unroll
        for (int j = 0; j < kRun; ++j) {
            const int b = threadIdx.x * kRun + j;
            c[j] = b < kCoarseBins ? __ldcg(hist + b) : 0ull;
        }
        scan();
    }

    __device__ void load_u32(const uint32_t* hist) {          // global, through L2
#pragma unroll
        for (int j = 0; j < kRun; ++j) {
            const int b = threadIdx.x * kRun + j;
            c[j] = b < kCoarseBins ? __ldcg(hist + b) : 0ull;
        }
        scan();
    }

    __device__ void load_shared(const uint32_t* hist) {
#pragma unroll
        for (int j = 0; j < kRun; ++j) {
            const int b = threadIdx.x * kRun + j;
            c[j] = b < kCoarseBins ? hist[b] : 0ull;
        }
        scan();
    }

    __device__ void scan() {
        __shared__ unsigned long long warp_sum[THREADS / 32];
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        run = 0;
#pragma unroll
        for (int j = 0; j < kRun; ++j) run += c[j];
        unsigned long long incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const unsigned long long o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) warp_sum[warp] = incl;
        __syncthreads();
        unsigned long long before = 0;
        total = 0;
#pragma unroll
        for (int w = 0; w < THREADS / 32; ++w) {
            before += w < warp ? warp_sum[w] : 0ull;
            total += warp_sum[w];
        }
        excl = before + incl - run;
        __syncthreads();
    }

    // true in exactly the one thread whose run holds rank r (1 <= r <= total): the bin
    // and the count of keys in the bins before it
    __device__ bool find(unsigned long long r, int& bin, unsigned long long& below) const {
        if (!(excl < r && r <= excl + run)) return false;
        unsigned long long cum = excl;
        bin = -1;
#pragma unroll
        for (int j = 0; j < kRun; ++j) {
            if (bin < 0) {
                if (r <= cum + c[j]) bin = threadIdx.x * kRun + j;
                else cum += c[j];
            }
        }
        below = cum;
        return true;
    }
};

// The coarse histogram of the active keys of slices first, first + stride, ...
// below `slices`, visited by block b at b, b + grid, ... (integer counts, so the
// order does not matter): per block in shared memory, then added to `hist`.
template <bool VEC>
__device__ void coarse_histogram(const float* nw, const float* od, const uint8_t* mask, int64_t N,
                                 int64_t slices, int64_t stride, unsigned long long* hist) {
    __shared__ uint32_t h[kCoarseBins];
    for (int i = threadIdx.x; i < kCoarseBins; i += kAuditThreads) h[i] = 0u;
    __syncthreads();
    uint32_t n_zero = 0;
#pragma unroll 1
    for (int64_t i = blockIdx.x; i * stride < slices; i += gridDim.x) {
        float4 x[kVec], y[kVec];
        uint32_t m[kVec];
        load_slice<VEC>(nw, od, mask, N, i * stride * kSlice, x, y, m);
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const float xs[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
            const float ys[4] = {y[j].x, y[j].y, y[j].z, y[j].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool act = ((m[j] >> (8 * e)) & 0xffu) != 0u;
                const uint32_t bits = __float_as_uint(xs[e] - ys[e]) & 0x7fffffffu;
                n_zero += (act && bits == 0u) ? 1u : 0u;
                if (act && bits != 0u) atomicAdd(&h[coarse_bin_nonzero(bits)], 1u);
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) n_zero += __shfl_down_sync(0xffffffffu, n_zero, off);
    if ((threadIdx.x & 31) == 0 && n_zero != 0u) atomicAdd(&h[kCoarseZero], n_zero);
    __syncthreads();
    for (int i = threadIdx.x; i < kCoarseBins; i += kAuditThreads)
        if (h[i] != 0u) atomicAdd(&hist[i], static_cast<unsigned long long>(h[i]));
}

// Sample slices: every K-th, kSampleSlices to 2 kSampleSlices - 1 of them (every
// slice of a batch of fewer than 2 kSampleSlices slices), one block each.
constexpr int64_t kSampleSlices = 128;
// Half-width of a window in standard deviations of a sample rank (plus 16 ranks).
// For a sample that represents the batch a rank leaves its window with probability
// below 1e-4; the fallback then keeps the result exact.
constexpr double kWindowSigmas = 4.0;

inline int64_t ext_sample_stride(int64_t slices) {
    return slices > kSampleSlices ? slices / kSampleSlices : 1;
}

// The sample's coarse histogram, per block in shared memory, then added to `shist`
// (cleared before the launch); the last block to finish (an integer ticket) sets the
// windows.  On the side the blocks clear the exact histogram of the fallback and the
// select histograms (nothing reads either before this kernel has finished).
template <bool VEC>
__global__ void __launch_bounds__(kAuditThreads)
    audit_ext_sample(const float* __restrict__ nw, const float* __restrict__ od,
                     const uint8_t* __restrict__ mask, int64_t N, int64_t stride,
                     uint32_t* __restrict__ shist, unsigned* __restrict__ ticket,
                     unsigned long long* __restrict__ hist, uint32_t* __restrict__ sel_hist,
                     ExtSelect* __restrict__ sel) {
    asm volatile("griddepcontrol.launch_dependents;");
    __shared__ uint32_t h[kCoarseBins];
    for (int i = threadIdx.x; i < kCoarseBins; i += kAuditThreads) h[i] = 0u;
    {
        const int g = blockIdx.x * kAuditThreads + threadIdx.x;
        const int all = gridDim.x * kAuditThreads;
        for (int i = g; i < kCoarseBins; i += all) hist[i] = 0ull;
        for (int i = g; i < kSelPasses * 3 * kSelBins; i += all) sel_hist[i] = 0u;
    }
    __syncthreads();
    const int64_t slices = (N + kSlice - 1) / kSlice;
    uint32_t n_zero = 0;
#pragma unroll 1
    for (int64_t i = blockIdx.x; i * stride < slices; i += gridDim.x) {
        float4 x[kVec], y[kVec];
        uint32_t m[kVec];
        load_slice<VEC>(nw, od, mask, N, i * stride * kSlice, x, y, m);
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const float xs[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
            const float ys[4] = {y[j].x, y[j].y, y[j].z, y[j].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool act = ((m[j] >> (8 * e)) & 0xffu) != 0u;
                const uint32_t bits = __float_as_uint(xs[e] - ys[e]) & 0x7fffffffu;
                n_zero += (act && bits == 0u) ? 1u : 0u;
                if (act && bits != 0u) atomicAdd(&h[coarse_bin_nonzero(bits)], 1u);
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) n_zero += __shfl_down_sync(0xffffffffu, n_zero, off);
    if ((threadIdx.x & 31) == 0 && n_zero != 0u) atomicAdd(&h[kCoarseZero], n_zero);
    __syncthreads();
    for (int i = threadIdx.x; i < kCoarseBins; i += kAuditThreads)
        if (h[i] != 0u) atomicAdd(&shist[i], h[i]);
    __shared__ bool s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    BinScan<kAuditThreads> bs;
    bs.load_u32(shist);
    const unsigned long long sa = bs.total;   // active keys in the sample
    // window ends in sample ranks; an end outside [1, sa] opens the window to that side
    __shared__ int s_bin[3][2];
    if (threadIdx.x < 3) {
        s_bin[threadIdx.x][0] = kCoarseZero;
        s_bin[threadIdx.x][1] = kCoarseHigh;
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 3; ++q) {
        if (sa == 0ull) break;
        const double pf = pct_of(q) / 100.0;
        const long long r = static_cast<long long>((pct_of(q) * sa + 99) / 100);
        const long long w = static_cast<long long>(
                                ceil(kWindowSigmas * sqrt(static_cast<double>(sa) * pf * (1.0 - pf)))) +
                            16;
        int bin;
        unsigned long long below;
        if (r - w >= 1 && bs.find(static_cast<unsigned long long>(r - w), bin, below))
            s_bin[q][0] = bin;
        if (r + w <= static_cast<long long>(sa) &&
            bs.find(static_cast<unsigned long long>(r + w), bin, below))
            s_bin[q][1] = bin;
    }
    __syncthreads();
    if (threadIdx.x < 3) {
        const int q = threadIdx.x;
        uint32_t lo, hi, lo2, hi2;
        coarse_bin_range(s_bin[q][0], lo, hi);
        coarse_bin_range(s_bin[q][1], lo2, hi2);
        sel->win_lo[q] = lo;
        sel->win_hi[q] = hi2;
        sel->fallback[q] = 0;
    }
    if (threadIdx.x == 0) sel->need_fallback = 0;
}

// The extended audit's pass over all slices (see above); the partition of the
// slices is the base audit's with at most kExtMaxBlocks blocks.

template <bool VEC>
__global__ void __launch_bounds__(kAuditThreads, 3)
    audit_ext_main(const float* __restrict__ nw, const float* __restrict__ od,
                   const uint8_t* __restrict__ mask, int64_t N, float clip_lo, float clip_hi,
                   ExtPartial* __restrict__ out, const ExtSelect* __restrict__ sel,
                   uint32_t* __restrict__ cand, uint32_t* __restrict__ wn) {
    asm volatile("griddepcontrol.wait;" ::: "memory");       // the windows
    asm volatile("griddepcontrol.launch_dependents;");
    __shared__ uint32_t skeys[kAuditV3PerThread][kAuditThreads];
    const ExtGeom g(N);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t wr = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
    ExtSlice x;
    x.skeys = skeys;
    x.one = (blockDim.x >> 30) | 1u;
    x.neg_one = 0u - x.one;
#pragma unroll
    for (int q = 0; q < 3; ++q) {
        x.lo[q] = sel->win_lo[q];
        x.span[q] = sel->win_hi[q] - x.lo[q];
        x.neg_lo[q] = 0ull - x.lo[q];
        x.neg_size[q] = 0ull - (static_cast<uint64_t>(x.span[q]) + 1ull);
    }
    x.clip_lo = clip_lo;
    x.clip_hi = clip_hi;
    x.cand = cand + wr * g.capw;
    x.qstride = g.qstride;
    RunAcc r;
    DFloat sabs{0.f, 0.f};
    int clip = 0;
    int visited = 0;
#pragma unroll 1
    for (int64_t sl = blockIdx.x; sl < g.slices; sl += gridDim.x) {
        const int64_t base = sl * kSlice;
        ThreadAcc a;
        load_and_visit_slice<VEC, true>(nw, od, mask, N, base, r.best_key, a, &x);
        r.add_slice(a, base);
        sabs = df_add(sabs, DFloat{x.sabs, 0.f});
        clip += x.clip;
        ++visited;
    }
    if (lane == 0) {
#pragma unroll
        for (int q = 0; q < 3; ++q) wn[q * kWnStride + wr] = x.n[q];
    }
    // the block's partial: the base audit's tree, then the same tree for |d|, the clips
    // and the counts below the windows (the thread's inactive elements, counted below
    // every window as key 0, taken off)
    const long long inactive = static_cast<long long>(visited) * kAuditV3PerThread - r.count;
    long long below[3] = {x.below[0] - inactive, x.below[1] - inactive, x.below[2] - inactive};
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        DFloat y;
        y.hi = __shfl_down_sync(0xffffffffu, sabs.hi, off);
        y.lo = __shfl_down_sync(0xffffffffu, sabs.lo, off);
        const int c = __shfl_down_sync(0xffffffffu, clip, off);
        long long b[3];
#pragma unroll
        for (int q = 0; q < 3; ++q) b[q] = __shfl_down_sync(0xffffffffu, below[q], off);
        if (lane + off < 32) {
            sabs = df_add(sabs, y);
            clip += c;
#pragma unroll
            for (int q = 0; q < 3; ++q) below[q] += b[q];
        }
    }
    __shared__ DFloat w_abs[kWarps];
    __shared__ int w_clip[kWarps];
    __shared__ long long w_below[kWarps][3];
    if (lane == 0) {
        w_abs[warp] = sabs;
        w_clip[warp] = clip;
#pragma unroll
        for (int q = 0; q < 3; ++q) w_below[warp][q] = below[q];
    }
    const AuditPartial bp = block_partial(r);      // its barrier also orders the writes above
    if (threadIdx.x == 0) {
        DFloat sa = w_abs[0];
        int64_t cl = w_clip[0];
        int64_t bl[3] = {w_below[0][0], w_below[0][1], w_below[0][2]};
#pragma unroll
        for (int w = 1; w < kWarps; ++w) {
            sa = df_add(sa, w_abs[w]);
            cl += w_clip[w];
#pragma unroll
            for (int q = 0; q < 3; ++q) bl[q] += w_below[w][q];
        }
        ExtPartial ep;
        ep.base = bp;
        ep.sum_abs = sa;
        ep.clip = cl;
#pragma unroll
        for (int q = 0; q < 3; ++q) ep.below[q] = bl[q];
        out[blockIdx.x] = ep;
    }
}

// One block: the fixed-order merge of the partials into the result; each
// percentile's rank, checked against its window.
__global__ void __launch_bounds__(kMergeThreads)
    audit_ext_merge(const ExtPartial* __restrict__ parts, int64_t num_parts,
                    const int64_t* __restrict__ seq_offsets, int64_t num_seqs,
                    rlk_audit_ext_t* __restrict__ result, ExtSelect* __restrict__ sel,
                    const uint32_t* __restrict__ wn) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    Acc a = empty_acc();
    DFloat sa{0.f, 0.f};
    int64_t cl = 0;
    int64_t bl[3] = {0, 0, 0};
    // ascending partials per thread, loaded in batches (as in the base audit's merge)
    auto fold = [&](const ExtPartial& p) {
        merge(a, to_acc(p.base));
        sa = df_add(sa, p.sum_abs);
        cl += p.clip;
#pragma unroll
        for (int q = 0; q < 3; ++q) bl[q] += p.below[q];
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
    // the candidates of each list: the warps' counts (integers: any order)
    int64_t nc[3] = {0, 0, 0};
    for (int64_t k = threadIdx.x; k < num_parts * kWarps; k += kMergeThreads) {
#pragma unroll
        for (int q = 0; q < 3; ++q) nc[q] += wn[q * kWnStride + k];
    }
    a = block_reduce<kMergeThreads>(a);
    __shared__ DFloat s_abs[kMergeThreads / 32];
    __shared__ long long s_clip[kMergeThreads / 32];
    __shared__ long long s_below[kMergeThreads / 32][3];
    __shared__ long long s_nc[kMergeThreads / 32][3];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // the same fixed tree for the extra sums (the counts are integers)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        DFloat x;
        x.hi = __shfl_down_sync(0xffffffffu, sa.hi, off);
        x.lo = __shfl_down_sync(0xffffffffu, sa.lo, off);
        const long long z = __shfl_down_sync(0xffffffffu, static_cast<long long>(cl), off);
        long long b[3], c[3];
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            b[q] = __shfl_down_sync(0xffffffffu, static_cast<long long>(bl[q]), off);
            c[q] = __shfl_down_sync(0xffffffffu, static_cast<long long>(nc[q]), off);
        }
        if (lane + off < 32) {
            sa = df_add(sa, x);
            cl += z;
#pragma unroll
            for (int q = 0; q < 3; ++q) {
                bl[q] += b[q];
                nc[q] += c[q];
            }
        }
    }
    if (lane == 0) {
        s_abs[warp] = sa;
        s_clip[warp] = cl;
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            s_below[warp][q] = bl[q];
            s_nc[warp][q] = nc[q];
        }
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    for (int w = 1; w < kMergeThreads / 32; ++w) {
        s_abs[0] = df_add(s_abs[0], s_abs[w]);
        s_clip[0] += s_clip[w];
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            s_below[0][q] += s_below[w][q];
            s_nc[0][q] += s_nc[w][q];
        }
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
    int need = 0;
    for (int q = 0; q < 3; ++q) {
        const int64_t rank = (pct_of(q) * a.count + 99) / 100;   // nearest rank, 1-based (0: none)
        const int64_t below = s_below[0][q];
        const int64_t ncq = s_nc[0][q];
        sel->rank[q] = rank;
        SelState st;
        if (rank <= 0) {
            st = window_state(1u, 1u, 0);                  // done; NaN stays
        } else if (below < rank && rank <= below + ncq) {
            st = window_state(sel->win_lo[q], sel->win_hi[q], rank - below);
        } else {
            st = window_state(1u, 1u, 0);                  // replaced by the fallback
            sel->fallback[q] = 1;
            need = 1;
        }
        sel->st[0][q] = st;
    }
    sel->need_fallback = need;
}

// Fallback, step 1 (returns at once unless some window missed its rank): the exact
// coarse histogram of all keys.
template <bool VEC>
__global__ void __launch_bounds__(kAuditThreads)
    audit_ext_fallback_hist(const float* __restrict__ nw, const float* __restrict__ od,
                            const uint8_t* __restrict__ mask, int64_t N,
                            unsigned long long* __restrict__ hist,
                            const ExtSelect* __restrict__ sel) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    if (sel->need_fallback == 0) return;
    const int64_t slices = (N + kSlice - 1) / kSlice;
    coarse_histogram<VEC>(nw, od, mask, N, slices, 1, hist);
}

// Fallback, step 2: every block finds the coarse bin of each missed rank (block 0
// stores the selection state), then the keys of those bins replace those lists,
// with the main pass's blocks, slices and warp ranges.
template <bool VEC>
__global__ void __launch_bounds__(kAuditThreads, 3)
    audit_ext_fallback_collect(const float* __restrict__ nw, const float* __restrict__ od,
                               const uint8_t* __restrict__ mask, int64_t N,
                               const unsigned long long* __restrict__ hist,
                               ExtSelect* __restrict__ sel, uint32_t* __restrict__ cand,
                               uint32_t* __restrict__ wn) {
    __shared__ int s_bin[3];
    __shared__ unsigned long long s_below[3];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    if (sel->need_fallback == 0) return;
    if (threadIdx.x < 3) {
        s_bin[threadIdx.x] = -1;
        s_below[threadIdx.x] = 0ull;
    }
    BinScan<kAuditThreads> bs;
    bs.load(hist);                                   // its barriers order the writes above
    for (int q = 0; q < 3; ++q) {
        int bin;
        unsigned long long below;
        if (sel->fallback[q] && bs.find(static_cast<unsigned long long>(sel->rank[q]), bin, below)) {
            s_bin[q] = bin;
            s_below[q] = below;
        }
    }
    __syncthreads();
    __shared__ uint32_t skeys[kAuditV3PerThread][kAuditThreads];
    const ExtGeom g(N);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t wr = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
    ExtSlice x;
    x.skeys = skeys;
    x.one = (blockDim.x >> 30) | 1u;
    x.neg_one = 0u - x.one;
    bool redo[3];
#pragma unroll
    for (int q = 0; q < 3; ++q) {
        x.lo[q] = 0xffffffffu;                        // an empty window: no key reaches it
        x.span[q] = 0u;
        redo[q] = s_bin[q] >= 0;
        if (redo[q]) {
            uint32_t lo, hi;
            coarse_bin_range(s_bin[q], lo, hi);
            const SelState st = window_state(lo, hi, sel->rank[q] - static_cast<int64_t>(s_below[q]));
            if (blockIdx.x == 0 && threadIdx.x == 0) {
                sel->st[0][q] = st;
                sel->win_lo[q] = lo;
                sel->win_hi[q] = hi;
            }
            x.lo[q] = lo;
            x.span[q] = hi - lo;
        }
        x.neg_lo[q] = 0ull - x.lo[q];
        x.neg_size[q] = 0ull - (static_cast<uint64_t>(x.span[q]) + 1ull);
    }
    x.clip_lo = -INFINITY;
    x.clip_hi = INFINITY;
    x.cand = cand + wr * g.capw;
    x.qstride = g.qstride;
#pragma unroll 1
    for (int64_t sl = blockIdx.x; sl < g.slices; sl += gridDim.x) {
        ThreadAcc a;
        load_and_visit_slice<VEC, true>(nw, od, mask, N, sl * kSlice, 0xffffffffu, a, &x);
    }
    if (lane == 0) {
#pragma unroll
        for (int q = 0; q < 3; ++q)
            if (redo[q]) wn[q * kWnStride + wr] = x.n[q];
    }
}

// The select step after radix pass p of percentile q: the digit whose bin holds
// the rank (an exclusive scan of the 2^bits counts, exact), appended to the known
// bits.  Run identically by every block of the next pass and by the final step.
__device__ void sel_step(int q, int p, const uint32_t* __restrict__ sel_hist,
                         SelState& st) {
    __shared__ unsigned long long warp_sum[kAuditThreads / 32];
    __shared__ uint32_t s_digit;
    __shared__ int64_t s_rank;
    int shift, bits;
    sel_digit(st.vbits, p, shift, bits);
    if (st.done || bits == 0) return;                  // block-uniform
    if (threadIdx.x == 0) {                            // (always overwritten: the counts are exact)
        s_digit = 0u;
        s_rank = 1;
    }
    const int nb = 1 << bits;
    const int runl = nb > kAuditThreads ? nb / kAuditThreads : 1;    // 8, 4, 2 or 1
    const uint32_t* hq = sel_hist + (static_cast<int64_t>(p) * 3 + q) * kSelBins;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long c[8];
    unsigned long long run = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int b = threadIdx.x * runl + j;
        c[j] = (j < runl && b < nb) ? __ldcg(hq + b) : 0ull;
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
    sel_digit(st.vbits, p + 1, s2, b2);
    st.done = (p + 1 >= kSelPasses || b2 == 0) ? 1 : 0;
    __syncthreads();
}

// Radix pass p over each percentile's candidates (blockIdx.y = percentile): block x
// reads the ranges of main-pass blocks x, x + R, x + 2R, ... (R = gridDim.x, one
// wave; warp w the ranges of their warps w) and counts digit p of the candidates
// that match the bits known so far.  For p > 0 every block first repeats the select step of
// pass p - 1; block 0 stores its outcome.
constexpr int kRadixBlocks = 152;
constexpr int kRadixBatch = 8;

template <int P>
__global__ void __launch_bounds__(kAuditThreads)
    audit_ext_radix(ExtSelect* __restrict__ sel, const uint32_t* __restrict__ cand,
                    const uint32_t* __restrict__ wn, int64_t N,
                    uint32_t* __restrict__ sel_hist) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int q = blockIdx.y;
    SelState st = sel->st[P == 0 ? 0 : P - 1][q];
    if (P > 0) {
        sel_step(q, P - 1, sel_hist, st);
        if (blockIdx.x == 0 && threadIdx.x == 0) sel->st[P][q] = st;
    }
    if (st.done) return;                                // block-uniform
    const uint32_t kmask = st.kmask, kvalue = st.kvalue;
    int shift, bits;
    sel_digit(st.vbits, P, shift, bits);
    const uint32_t dmask = (1u << bits) - 1u;
    __shared__ uint32_t h[kSelBins];
    for (int i = threadIdx.x; i < kSelBins; i += kAuditThreads) h[i] = 0u;
    __syncthreads();
    const ExtGeom g(N);
    const int lane = threadIdx.x & 31;
    for (int64_t b = blockIdx.x; b < g.blocks; b += gridDim.x) {
        const int64_t wr = b * kWarps + (threadIdx.x >> 5);
        const int64_t n = wn[q * kWnStride + wr];
        const uint32_t* cq = cand + q * g.qstride + wr * g.capw;
        // kRadixBatch keys per lane loaded before any is counted, so their loads overlap
        for (int64_t base = 0; base < n; base += 32 * kRadixBatch) {
            uint32_t kk[kRadixBatch];
#pragma unroll
            for (int u = 0; u < kRadixBatch; ++u) {
                const int64_t i = base + u * 32 + lane;
                kk[u] = i < n ? cq[i] : 0u;             // 0: no key (keys start at 1)
            }
#pragma unroll
            for (int u = 0; u < kRadixBatch; ++u) {
                const uint32_t k = kk[u] - 1u;
                const bool match = kk[u] != 0u && (k & kmask) == kvalue;
                const uint32_t digit = (k >> shift) & dmask;
                // equal digits within the warp add up in one atomic (many equal keys are common)
                const unsigned act = __ballot_sync(0xffffffffu, match);
                if (match) {
                    const unsigned peers = __match_any_sync(act, digit);
                    if (lane == __ffs(peers) - 1) atomicAdd(&h[digit], __popc(peers));
                }
            }
        }
    }
    __syncthreads();
    uint32_t* gh = sel_hist + (static_cast<int64_t>(P) * 3 + q) * kSelBins;
    for (int i = threadIdx.x; i < (1 << bits); i += kAuditThreads)
        if (h[i] != 0u) atomicAdd(&gh[i], h[i]);
}

// The last select step; the selected |d| bits become p50 / p90 / p99.
__global__ void __launch_bounds__(kAuditThreads)
    audit_ext_finish(const ExtSelect* __restrict__ sel, const uint32_t* __restrict__ sel_hist,
                     rlk_audit_ext_t* __restrict__ result) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int q = 0; q < 3; ++q) {
        SelState st = sel->st[kSelPasses - 1][q];
        if (st.rank <= 0) continue;                      // no active token: NaN stays
        sel_step(q, kSelPasses - 1, sel_hist, st);
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

// extended audit workspace: partials | sample histogram (u32) and ticket (cleared
// by one memset) | the fallback's exact histogram | select state | select
// histograms | the warps' list lengths [3][kWnStride] | candidate lists
// [3][qstride] (uint32).  Nothing else in it has to start at zero: the sample
// kernel clears the other two histograms.
struct ExtLayout {
    size_t shist_off, ticket_off, hist_off, sel_off, selhist_off, wn_off, cand_off, total;
    explicit ExtLayout(int64_t N) {
        const ExtGeom g(N);
        shist_off = align_up(static_cast<size_t>(kExtMaxBlocks) * sizeof(ExtPartial), 256);
        ticket_off = shist_off + kCoarseBins * sizeof(uint32_t);
        hist_off = align_up(ticket_off + 16, 256);
        sel_off = align_up(hist_off + kCoarseBins * sizeof(unsigned long long), 256);
        selhist_off = align_up(sel_off + sizeof(ExtSelect), 256);
        wn_off = align_up(selhist_off + kSelPasses * 3 * kSelBins * sizeof(uint32_t), 256);
        cand_off = align_up(wn_off + 3 * static_cast<size_t>(kWnStride) * 4, 256);
        total = align_up(cand_off + 3 * static_cast<size_t>(g.qstride) * 4, 256) + 256;
    }
};

size_t audit_ext_workspace(int64_t N) { return ExtLayout(N).total; }

cudaError_t launch_audit_ext(const float* logp_new, const float* logp_old, const uint8_t* mask,
                             int64_t N, const int64_t* seq_offsets, int64_t num_seqs, float eps,
                             rlk_audit_ext_t* result, void* workspace, bool vec_ok, int sms,
                             cudaStream_t stream) {
    (void)sms;
    const ExtLayout lay(N);
    const ExtGeom geo(N);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    ExtPartial* parts = reinterpret_cast<ExtPartial*>(ws);
    uint32_t* shist = reinterpret_cast<uint32_t*>(ws + lay.shist_off);
    unsigned* ticket = reinterpret_cast<unsigned*>(ws + lay.ticket_off);
    unsigned long long* hist = reinterpret_cast<unsigned long long*>(ws + lay.hist_off);
    ExtSelect* sel = reinterpret_cast<ExtSelect*>(ws + lay.sel_off);
    uint32_t* sel_hist = reinterpret_cast<uint32_t*>(ws + lay.selhist_off);
    uint32_t* wn = reinterpret_cast<uint32_t*>(ws + lay.wn_off);
    uint32_t* cand = reinterpret_cast<uint32_t*>(ws + lay.cand_off);
    // the clip thresholds of |exp(d) - 1| > eps, rounded to fp32 once
    const double e = static_cast<double>(eps);
    const float clip_hi = static_cast<float>(std::log1p(e));
    const float clip_lo = e < 1.0 ? static_cast<float>(std::log1p(-e)) : -INFINITY;
    if (geo.slices == 0) {
        audit_ext_merge<<<1, kMergeThreads, 0, stream>>>(parts, 0, seq_offsets, num_seqs, result,
                                                         sel, wn);
        return cudaGetLastError();
    }
    const int64_t stride = ext_sample_stride(geo.slices);
    const unsigned blocks = static_cast<unsigned>(geo.blocks);
    cudaError_t err = cudaMemsetAsync(ws + lay.shist_off, 0, lay.ticket_off + 16 - lay.shist_off, stream);
    if (err != cudaSuccess) return err;
    const unsigned sgrid = static_cast<unsigned>((geo.slices + stride - 1) / stride);
    if (vec_ok)
        audit_ext_sample<true><<<sgrid, kAuditThreads, 0, stream>>>(
            logp_new, logp_old, mask, N, stride, shist, ticket, hist, sel_hist, sel);
    else
        audit_ext_sample<false><<<sgrid, kAuditThreads, 0, stream>>>(
            logp_new, logp_old, mask, N, stride, shist, ticket, hist, sel_hist, sel);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    // the rest: each launch may begin while the previous one runs, and waits for it
    // in-kernel (programmatic dependent launch)
    auto dep = [&](auto kernel, dim3 grid, unsigned threads, auto... args) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(threads);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kernel, args...);
    };
#define RLK_TRY(x)                               \
    do {                                         \
        const cudaError_t e_ = (x);              \
        if (e_ != cudaSuccess) return e_;        \
    } while (0)
    const ExtSelect* csel = sel;
    const ExtPartial* cparts = parts;
    const unsigned long long* chist = hist;
    const uint32_t* cwn = wn;
    const uint32_t* ccand = cand;
    const int64_t nparts = geo.blocks;
    if (vec_ok) {
        RLK_TRY(dep(audit_ext_main<true>, dim3(blocks), kAuditThreads, logp_new, logp_old, mask, N,
                    clip_lo, clip_hi, parts, csel, cand, wn));
    } else {
        RLK_TRY(dep(audit_ext_main<false>, dim3(blocks), kAuditThreads, logp_new, logp_old, mask, N,
                    clip_lo, clip_hi, parts, csel, cand, wn));
    }
    RLK_TRY(dep(audit_ext_merge, dim3(1), kMergeThreads, cparts, nparts, seq_offsets, num_seqs,
                result, sel, cwn));
    if (vec_ok) {
        RLK_TRY(dep(audit_ext_fallback_hist<true>, dim3(blocks), kAuditThreads, logp_new, logp_old,
                    mask, N, hist, csel));
        RLK_TRY(dep(audit_ext_fallback_collect<true>, dim3(blocks), kAuditThreads, logp_new,
                    logp_old, mask, N, chist, sel, cand, wn));
    } else {
        RLK_TRY(dep(audit_ext_fallback_hist<false>, dim3(blocks), kAuditThreads, logp_new, logp_old,
                    mask, N, hist, csel));
        RLK_TRY(dep(audit_ext_fallback_collect<false>, dim3(blocks), kAuditThreads, logp_new,
                    logp_old, mask, N, chist, sel, cand, wn));
    }
    const dim3 rgrid(static_cast<unsigned>(std::min<int64_t>(geo.blocks, kRadixBlocks)), 3);
    RLK_TRY(dep(audit_ext_radix<0>, rgrid, kAuditThreads, sel, ccand, cwn, N, sel_hist));
    RLK_TRY(dep(audit_ext_radix<1>, rgrid, kAuditThreads, sel, ccand, cwn, N, sel_hist));
    RLK_TRY(dep(audit_ext_radix<2>, rgrid, kAuditThreads, sel, ccand, cwn, N, sel_hist));
    const uint32_t* csh = sel_hist;
    RLK_TRY(dep(audit_ext_finish, dim3(1), kAuditThreads, csel, csh, result));
#undef RLK_TRY
    return cudaSuccess;
}

}  // namespace rlk
