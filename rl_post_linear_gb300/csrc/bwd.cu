// bwd.cu -- chunked-recompute backward of the fused linear log-prob.
//
// "RL-Kernel Roadmap (2026)", P0.2: the backward recomputes tiles to trade
// compute for memory instead of storing full logits or probabilities.
// "RL-Kernel integration roadmap for vime", linear_logp: dlogits live in
// operator-owned workspace; the operator returns full gradients.
//
// With g_t = dL/dlogp_t, k = log2(e)/T and lse2_t = lse_t log2(e), the
// gradient of the logits is G[t,v] = (g_t / T)(delta_{v,y_t} - p[t,v]),
// p[t,v] = 2^(S[t,v] k - lse2_t) (S recomputed, fp32).  It is applied as
//   dS[t,v] = -(g_t / T) p[t,v]                       (bf16, v not y_t, a_t)
//   dS[t,y] = 0,  dS[t,a] = (g_t / T)(1 - p[t,a])     (bf16)
//   dh_t    = bf16( sum_c (dS_c W_c)_t + (g_t / T)(1 - p_y) W[y_t] - (g_t / T) W[a_t] )
//   dW_v    = bf16( (dS^T h)_v + sum_{y_t = v} (g_t / T)(1 - p_y) h_t
//                               - sum_{a_t = v} (g_t / T) h_t )
// where a_t is the row's dominant non-target class (p > 1/2), if any.  The
// large parts of the two entries that can dominate a row are added in fp32 in
// the epilogues, with 1 - p = -expm1(log p): in bf16 dS the target's g/T part
// (flat softmax) would cost as much accuracy as the final rounding of the
// outputs, and g (1 - p) / T written as a difference (a confident policy,
// p -> 1) would lose its leading digits.
//
// The vocabulary is walked in fixed chunks of kBwdChunk columns, ascending.
// For each chunk c three tcgen05 GEMM roles run:
//   DsPolicy  S_c = h W_c^T (K = H) -> dS_c [N, chunk] bf16 workspace
//   DhPolicy  dS_c W_c (K = chunk)  -> dh_acc [N, H] fp32 (+= previous chunks;
//             the last chunk adds the target term and rounds to bf16)
//   DwPolicy  dS_c^T h (K = N)      -> dW rows of chunk c, plus target terms
// A masked batch is first compacted to its active rows (ascending token order,
// the forward's gather): h, dS and dh_acc rows are then compacted rows, the K
// loop of dW runs over ceil(N_active / 64) blocks, and each dh row is written at
// its token; the inactive tokens' dh rows are zeroed apart.
// Each role is one persistent launch per chunk, in that order (measured faster
// than putting roles of neighbouring chunks side by side in one launch: alone,
// each role keeps its L2 working set), on CTA pairs with 256 x 256 tiles.
// For the entropy and KL backwards, whose gradients have no fp32 part that
// dominates a row, dS is stored as two bf16 planes, hi = bf16(dS) and
// lo = bf16(dS - hi); the dh and dW K loops run over both planes against the
// same W (or h) blocks, so dS enters the products with about 16 significant
// bits.
// None of the reductions is split or done with atomics: dh_t depends only on
// row t's inputs and the fixed chunk boundaries, so it is batch invariant;
// dW is reproducible bit for bit.
//
// The target terms of dW need, for each vocab row v, the tokens with y_t = v
// in ascending t: the tokens sorted by the unique 64-bit key (y_t, t), y_t
// taken as V for inactive rows and invalid targets.  Two launches, no atomics
// on positions: each block sorts a tile of 2048 keys in shared memory
// (Batcher's bitonic network); then each key's place in the whole list is its
// place in its own tile plus, for every other tile, the number of that tile's
// keys below it (a binary search).  Keys are unique, so the result is the one
// sorted order whatever the schedule.
#include <cuda_bf16.h>

#include "gemm.cuh"

namespace rlk {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// The rounding residues of a pair packed by pack_bf16x2: bf16(d - bf16(d)) of
// both values.  d - bf16(d) is exact in fp32, so hi + lo carries d to about 16
// significant bits.
__device__ __forceinline__ uint32_t pack_lo_bf16x2(float d0, float d1, uint32_t hi) {
    const float h0 = __uint_as_float(hi << 16);
    const float h1 = __uint_as_float(hi & 0xffff0000u);
    return pack_bf16x2(d0 - h0, d1 - h1);
}

__device__ __forceinline__ bool row_live(const int64_t* targets, const uint8_t* mask, int t, int N,
                                         int V, int64_t& y) {
    y = 0;
    if (t >= N) return false;
    if (mask != nullptr && mask[t] == 0) return false;
    y = targets[t];
    return y >= 0 && y < V;
}

// Rows of a masked batch compacted to its active tokens (ascending): GEMM row i
// is token rows[i] for i < *n_rows.  Both nullptr: rows are tokens.
struct RowMap {
    const int* rows;
    const int* n_rows;
    __device__ int count(int N) const { return n_rows != nullptr ? *n_rows : N; }
    // at least one tile: with no active row, the dS GEMM still zeroes the rows that
    // the dW GEMM's (single) K block reads
    __device__ int tiles(int N) const { return (max(count(N), 1) + kUnitM - 1) / kUnitM; }
    __device__ int token(int i) const { return rows != nullptr ? rows[i] : i; }
};

__device__ __forceinline__ void bf16x8_to_f32(uint4 v, float* out) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        out[2 * i] = __uint_as_float(w[i] << 16);
        out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// ----------------------------------------------------------------------------- dS_c

// ENT adds the entropy gradient: with Ez = lse - entropy (= E_p[z]),
//   dS = p (c1 + c2 S),  c1 = -(g - gH Ez) / T,  c2 = -gH / T^2,
// i.e. -(p/T) (g + gH (S/T - Ez)), the entropy's dH/dz = -p (z - E[z]).
template <bool ENT>
struct DsPolicyT : SingleRole<false, false> {   // h [N,H], W [V,H]: K-major
    static constexpr bool kCtaPair = true;       // 256-token tiles on a CTA pair
    // With ENT, dS is stored as a pair of bf16 planes per row, hi = bf16(dS) and
    // lo = bf16(dS - hi) (columns [kBwdChunk, 2 kBwdChunk) of the row), and the dh and
    // dW GEMMs run over both planes: the entropy gradient has no fp32 part that
    // dominates the row, so a single bf16 rounding of dS would cost as much accuracy
    // as the final rounding of the outputs.  Rows with gH = 0 keep lo = 0 and so give
    // the logp-only backward's dh rows bit for bit.
    static constexpr int kLd = ENT ? 2 * kBwdChunk : kBwdChunk;   // dS row stride

    const int64_t* targets;
    const uint8_t* mask;
    const float* grad;
    const float* grad_ent;   // ENT only
    const float* ent;        // ENT only
    const float* lse;
    __nv_bfloat16* ds;    // [N][kBwdChunk]
    float* ycoef;         // [N]: 1 - p_y of each live row, written by the tile holding y
    int* dom;             // [N]: the row's dominant non-target class (p > 1/2), else -1
    float* dcoef;         // [N]: that class's fp32 gradient coefficient, -g/T
    int* dom_flag;        // set to 1 when some row's dominant class lies in this chunk
    int64_t y_off;        // global id of this weight block's first row (0 unsharded)
    int V_global;         // vocabulary size (target validity)
    RowMap rm;            // compaction of a masked batch (dS rows are compacted rows)
    int N, V, c0, num_m, num_n, kblocks;   // V: rows of this weight block
    float k, temp;

    __device__ int num_units() const { return rm.tiles(N) * num_n; }
    __device__ int k_blocks(int) const { return kblocks; }
    __device__ int tiles_in_unit(int) const { return 1; }
    // unit -> (row tile m, vocab tile n of the chunk), row tiles grouped
    __device__ void unit(int u, int& m, int& n) const {
        grouped_unit(u, rm.tiles(N), num_n, kRasterTokenRows / kUnitM, m, n);
    }
    __device__ void coords(int u, int, int& a_mn, int& a_k, int& b_mn, int& b_k) const {
        int m, n;
        unit(u, m, n);
        a_mn = m * kUnitM;
        a_k = 0;
        b_mn = c0 + n * kTileV;
        b_k = 0;
    }

    struct EpiState {
        float coef, c2, lse2;
        float coef_y;         // ENT: the target entry's coefficient without the -g/T part
        float gt;             // g / T
        int64_t ycol;         // target column relative to the chunk
        int t;                // the row's token
        bool live;
        bool lo;              // ENT: the row stores the lo plane of dS (gH != 0)
    };

    __device__ void epi_begin(int u, int row, EpiState& st) const {
        int m, n;
        unit(u, m, n);
        const int i = m * kUnitM + row;
        const int t = i < rm.count(N) ? rm.token(i) : N;
        st.t = t;
        int64_t y;
        st.live = row_live(targets, mask, t, N, V_global, y);
        st.lse2 = st.live ? lse[t] * kLog2e : 0.f;
        st.ycol = y - y_off - c0;       // outside [0, 32 * 8) unless y is in this chunk
        st.coef_y = 0.f;
        st.lo = false;
        st.gt = st.live ? __fdiv_rn(grad[t], temp) : 0.f;
        if constexpr (ENT) {
            const float gh = st.live ? grad_ent[t] : 0.f;
            st.lo = gh != 0.f;
            const float ez = st.live ? lse[t] - ent[t] : 0.f;
            st.coef = st.live ? -__fdiv_rn(fmaf(-gh, ez, grad[t]), temp) : 0.f;
            st.c2 = st.live ? -__fdiv_rn(gh, temp * temp) : 0.f;
            st.coef_y = st.live ? __fdiv_rn(gh * ez, temp) : 0.f;
        } else {
            st.coef = st.live ? -__fdiv_rn(grad[t], temp) : 0.f;
            st.c2 = 0.f;
        }
    }

    __device__ void epi_tile(int u, int, int row, uint32_t taddr, EpiState& st) const {
        int m, n;
        unit(u, m, n);
        const int i = m * kUnitM + row;          // dS row (compacted row)
        const int t = st.t;                      // its token
#pragma unroll 1
        for (int cc = 0; cc < kTileV / 32; ++cc) {
            uint32_t r[32];
            tmem_load_32(taddr + cc * 32, r);
            if (i >= N) continue;
            const int col = n * kTileV + cc * 32;   // column inside the chunk
            const int vb = c0 + col;
            // The target entry: its -g p_y / T part stays out of dS, and the dh / dW
            // epilogues add g (1 - p_y) / T in fp32 instead of g / T.  1 - p_y comes from
            // expm1 of log p_y, so a dominant target (p_y -> 1) keeps its small gradient
            // g (1 - p_y) / T to fp32 accuracy rather than as a difference of two bf16-sized
            // terms.  (ENT keeps the entropy part of the entry in dS.)
            const int64_t yc = st.ycol - col;
            int yi = 32;                              // no target in this slice
            float dy = 0.f;
            float x[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]);
            if (st.live && yc >= 0 && yc < 32) {
                yi = static_cast<int>(yc);
                const float sy = select32(x, yi);
                const float l2 = fmaf(sy, k, -st.lse2);          // log2 p_y
                ycoef[t] = -expm1f(l2 * kLn2);
                if constexpr (ENT) dy = fmaf(st.c2, sy, st.coef_y) * ex2_approx(l2);
            }
            // A dominant non-target entry is split the same way: G_a = -g/T + (g/T)(1 - p_a)
            // (+ its entropy part); dS keeps the small second part, and the dh / dW
            // epilogues add -g/T in fp32 for the class recorded in dom.  "Dominant" is
            // p_a > 2^-0.99 = 0.5035: two entries of a row cannot both pass, even with the
            // fp32 error of p, so dom has one writer.
            int ai = 32;                              // no dominant entry in this slice
            float da = 0.f;
            const bool full = vb + 32 <= V;           // no column of the slice is past V
            if (st.live) {
                float cm = -INFINITY;
                if (full) {
                    cm = fmaxf(cm, max32(x));
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) cm = (vb + j < V) ? fmaxf(cm, x[j]) : cm;
                }
                const float l2 = fmaf(cm, k, -st.lse2);          // log2 of the slice's top p
                if (l2 > -0.99f) {
                    int idx = 31;
#pragma unroll
                    for (int j = 31; j >= 0; --j) idx = (x[j] == cm && vb + j < V) ? j : idx;
                    if (idx != yi) {
                        ai = idx;
                        dom[t] = vb + idx;
                        dcoef[t] = -st.gt;
                        atomicOr(dom_flag, 1);   // set by many rows
                        da = st.gt * -expm1f(l2 * kLn2);
                        if constexpr (ENT) da = fmaf(fmaf(st.c2, cm, st.coef_y), ex2_approx(l2), da);
                    }
                }
            }
            uint32_t packed[16];
            uint32_t packed_lo[ENT ? 16 : 1];
            if (full && yi == 32 && ai == 32 && st.live) {
                // the common slice: a live row, every column inside V, no target or
                // dominant entry to patch in (the same arithmetic as below, without the
                // selects)
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float s0 = x[2 * j];
                    const float s1 = x[2 * j + 1];
                    float c0 = st.coef, c1 = st.coef;
                    if constexpr (ENT) {
                        c0 = fmaf(st.c2, s0, st.coef);
                        c1 = fmaf(st.c2, s1, st.coef);
                    }
                    const float d0 = c0 * ex2_approx(fmaf(s0, k, -st.lse2));
                    const float d1 = c1 * ex2_approx(fmaf(s1, k, -st.lse2));
                    packed[j] = pack_bf16x2(d0, d1);
                    if constexpr (ENT)
                        packed_lo[j] = st.lo ? pack_lo_bf16x2(d0, d1, packed[j]) : 0u;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float s0 = x[2 * j];
                    const float s1 = x[2 * j + 1];
                    float c0 = st.coef, c1 = st.coef;
                    if constexpr (ENT) {
                        c0 = fmaf(st.c2, s0, st.coef);
                        c1 = fmaf(st.c2, s1, st.coef);
                    }
                    float d0 = (st.live && vb + 2 * j < V)
                                   ? c0 * ex2_approx(fmaf(s0, k, -st.lse2)) : 0.f;
                    float d1 = (st.live && vb + 2 * j + 1 < V)
                                   ? c1 * ex2_approx(fmaf(s1, k, -st.lse2)) : 0.f;
                    d0 = (yi == 2 * j) ? dy : ((ai == 2 * j) ? da : d0);
                    d1 = (yi == 2 * j + 1) ? dy : ((ai == 2 * j + 1) ? da : d1);
                    packed[j] = pack_bf16x2(d0, d1);
                    if constexpr (ENT)
                        packed_lo[j] = st.lo ? pack_lo_bf16x2(d0, d1, packed[j]) : 0u;
                }
            }
            uint4* dst = reinterpret_cast<uint4*>(ds + static_cast<size_t>(i) * kLd + col);
#pragma unroll
            for (int w = 0; w < 4; ++w)
                dst[w] = make_uint4(packed[4 * w], packed[4 * w + 1], packed[4 * w + 2],
                                    packed[4 * w + 3]);
            if constexpr (ENT) {
                uint4* dlo = reinterpret_cast<uint4*>(ds + static_cast<size_t>(i) * kLd +
                                                      kBwdChunk + col);
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    dlo[w] = make_uint4(packed_lo[4 * w], packed_lo[4 * w + 1],
                                        packed_lo[4 * w + 2], packed_lo[4 * w + 3]);
            }
        }
    }

    __device__ void epi_end(int, int, EpiState&) const {}
};

// ----------------------------------------------------------------------------- dS_c for KL
//
// Backward of L = sum_t g_t KL(p_t || q_t) + gr_t KL(q_t || p_t) with respect to
// the policy head only.  With l_v = log p_v - log q_v:
//   dKL(p||q)/dz_v = p_v (l_v - KL),   dKL(q||p)/dz_v = p_v - q_v,
//   dS[t,v] = ( g_t p_v (l_v - KL_t) + gr_t (p_v - q_v) ) / T          (bf16)
// Both logit tiles are recomputed (the mainloop's paired-tile mode: policy
// into one TMEM accumulator, reference into the other).  The entry of a
// dominant policy class (p > 2^-0.99, at most one per row) usually carries
// most of the row's gradient; it skips bf16 dS and reaches dh / dW through
// the same fp32 path as the logp backward's dominant classes (dom, dcoef and
// the per-chunk sorted list).  The dh and dW roles run without target terms.

struct DsKlMaps {
    CUtensorMap h, w, hr, wr;     // K-major; boxes {64,128} (each CTA of a pair loads 128 rows)
    CUtensorMap ds;               // dS [N, kLd] written by TMA stores, box {32, 32}, no swizzle
};

struct DsKlPolicy {
    using Maps = DsKlMaps;
    static constexpr bool kPairTiles = true;
    static constexpr bool kKRemap = false;
    static constexpr bool kCtaPair = true;    // 256-token units on a CTA pair
    static constexpr int kEpiWarps = 8;       // two column halves per row
    // Each epilogue warp stages its 32 rows x 32 columns of the hi and lo planes
    // (2 KiB each) in shared memory and writes them with two TMA stores, so that
    // the epilogue the MMA waits for issues no per-row global stores.
    static constexpr int kEpiSmemPerWarp = 4096;
    // dS as hi / lo bf16 planes (columns [0, kBwdChunk) and [kBwdChunk, 2 kBwdChunk) of
    // each row), which the dh and dW GEMMs both consume: the KL gradient has no fp32
    // part that dominates a row, so one bf16 rounding of dS would cost as much
    // accuracy as the final rounding of the outputs.
    static constexpr int kLd = 2 * kBwdChunk;

    const uint8_t* mask;
    const float* grad;        // d L / d KL(p||q), or nullptr
    const float* grad_rev;    // d L / d KL(q||p), or nullptr
    const float* lse;
    const float* lse_ref;
    const float* kl;
    __nv_bfloat16* ds;        // [N][kBwdChunk]
    int* dom;                 // [N] dominant policy class or -1
    float* dcoef;             // [N] its fp32 gradient entry
    int* dom_flag;            // set to 1 when some row's dominant class lies in this chunk
    int N, V, c0, num_m, num_n, kblocks, kblocks_r;
    float k, kr, temp;

    __device__ static void prefetch(const Maps& m) {
        prefetch_tensormap(&m.h);
        prefetch_tensormap(&m.w);
        prefetch_tensormap(&m.hr);
        prefetch_tensormap(&m.wr);
    }
    __device__ static const CUtensorMap* a_map(const Maps& m, int) { return &m.h; }
    __device__ static const CUtensorMap* b_map(const Maps& m, int) { return &m.w; }
    __device__ static const CUtensorMap* tile_a_map(const Maps& m, int, int q) {
        return (q & 1) ? &m.hr : &m.h;
    }
    __device__ static const CUtensorMap* tile_b_map(const Maps& m, int, int q) {
        return (q & 1) ? &m.wr : &m.w;
    }
    __device__ static bool a_mn(int) { return false; }
    __device__ static bool b_mn(int) { return false; }
    __device__ int k_blocks(int) const { return kblocks; }
    __device__ int tile_k_blocks(int, int q) const { return (q & 1) ? kblocks_r : kblocks; }

    __device__ int num_units() const { return num_m * num_n; }
    __device__ int tiles_in_unit(int) const { return 2; }
    __device__ void unit(int u, int& m, int& n) const {
        grouped_unit(u, num_m, num_n, kRasterTokenRows / kUnitM, m, n);
    }
    __device__ void coords(int u, int, int& a_mn, int& a_k, int& b_mn, int& b_k) const {
        int m, n;
        unit(u, m, n);
        a_mn = m * kUnitM;
        a_k = 0;
        b_mn = c0 + n * kTileV;
        b_k = 0;
    }

    struct EpiState {
        float lse2, lse2r, kl, gp, gq;
        float gpl, gpk;            // gp ln 2 and gp KL: g = p (gpl (l2p - l2q) - gpk) + gq (p - q)
        bool live;
    };

    __device__ void epi_begin(int u, int row, int, EpiState& st) const {
        int m, n;
        unit(u, m, n);
        const int t = m * kUnitM + row;
        st.live = t < N && (mask == nullptr || mask[t] != 0);
        st.lse2 = st.live ? lse[t] * kLog2e : 0.f;
        st.lse2r = st.live ? lse_ref[t] * kLog2e : 0.f;
        st.kl = (st.live && grad != nullptr) ? kl[t] : 0.f;
        st.gp = (st.live && grad != nullptr) ? __fdiv_rn(grad[t], temp) : 0.f;
        st.gq = (st.live && grad_rev != nullptr) ? __fdiv_rn(grad_rev[t], temp) : 0.f;
        st.gpl = st.gp * kLn2;
        st.gpk = st.gp * st.kl;
    }

    __device__ void epi_pair(const Maps& maps, int u, int, int row, int half, uint32_t tp,
                             uint32_t tr, EpiState& st, uint8_t* stage) const {
        int m, n;
        unit(u, m, n);
        const int t = m * kUnitM + row;
        const int lane = row & 31;
        const int t0 = t - lane;                    // the warp's first row
#pragma unroll 1
        for (int cc = half * (kTileV / 64); cc < (half + 1) * (kTileV / 64); ++cc) {
            uint32_t rp[32], rr[32];
            tmem_load_32x2(tp + cc * 32, rp, tr + cc * 32, rr);
            // rows past N compute zeros (not live); the TMA store drops them
            const int col = n * kTileV + cc * 32;   // column inside the chunk
            const int vb = c0 + col;
            // the slice's top policy entry, if it dominates the row
            int ai = 32;
            const bool full = vb + 32 <= V;             // no column of the slice is past V
            if (st.live) {
                float cm = -INFINITY;
                if (full) {
                    float xp[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) xp[j] = __uint_as_float(rp[j]);
                    cm = fmaxf(cm, max32(xp));
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        cm = (vb + j < V) ? fmaxf(cm, __uint_as_float(rp[j])) : cm;
                }
                if (fmaf(cm, k, -st.lse2) > -0.99f) {
                    int idx = 31;
#pragma unroll
                    for (int j = 31; j >= 0; --j)
                        idx = (__uint_as_float(rp[j]) == cm && vb + j < V) ? j : idx;
                    ai = idx;
                }
            }
            uint32_t packed[16], packed_lo[16];
            float gdom = 0.f;                           // the dominant entry's gradient
            if (full && ai == 32 && st.live) {
                // the common slice: a live row, every column inside V and no dominant
                // entry; the gradient grouped as p (gp ln2 (log2 p - log2 q) - gp KL) +
                // gq (p - q), two operations fewer an entry than below (identical heads
                // still give exactly 0)
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float d[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float s = __uint_as_float(rp[2 * j + e]);
                        const float r = __uint_as_float(rr[2 * j + e]);
                        const float l2p = fmaf(s, k, -st.lse2);     // log2 p
                        const float l2q = fmaf(r, kr, -st.lse2r);   // log2 q
                        const float p = ex2_approx(l2p), q = ex2_approx(l2q);
                        const float tt = fmaf(st.gpl, l2p - l2q, -st.gpk);
                        d[e] = fmaf(p, tt, st.gq * (p - q));
                    }
                    packed[j] = pack_bf16x2(d[0], d[1]);
                    packed_lo[j] = pack_lo_bf16x2(d[0], d[1], packed[j]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float d[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float s = __uint_as_float(rp[2 * j + e]);
                        const float r = __uint_as_float(rr[2 * j + e]);
                        const float l2p = fmaf(s, k, -st.lse2);     // log2 p
                        const float l2q = fmaf(r, kr, -st.lse2r);   // log2 q
                        const float p = ex2_approx(l2p), q = ex2_approx(l2q);
                        const float ell = (l2p - l2q) * kLn2;
                        const float g = fmaf(st.gp * p, ell - st.kl, st.gq * (p - q));
                        const bool is_dom = ai == 2 * j + e;        // fp32 path, not dS
                        gdom = is_dom ? g : gdom;
                        d[e] = (st.live && vb + 2 * j + e < V && !is_dom) ? g : 0.f;
                    }
                    packed[j] = pack_bf16x2(d[0], d[1]);
                    packed_lo[j] = pack_lo_bf16x2(d[0], d[1], packed[j]);
                }
            }
            if (ai < 32) {
                dom[t] = vb + ai;
                dcoef[t] = gdom;
                atomicOr(dom_flag, 1);   // set by many rows
            }
            // the slot is free once the previous slice's stores have read it
            if (lane == 0) bulk_wait_group_read0();
            __syncwarp();
            uint4* shi = reinterpret_cast<uint4*>(stage + lane * 64);
            uint4* slo = reinterpret_cast<uint4*>(stage + 2048 + lane * 64);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                shi[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                    packed[4 * i + 3]);
                slo[i] = make_uint4(packed_lo[4 * i], packed_lo[4 * i + 1], packed_lo[4 * i + 2],
                                    packed_lo[4 * i + 3]);
            }
            fence_proxy_async_smem();               // visible to the TMA engine
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(&maps.ds, stage, col, t0);
                tma_store_2d(&maps.ds, stage + 2048, kBwdChunk + col, t0);
                bulk_commit_group();
            }
        }
    }

    __device__ void epi_end(int, int, int, EpiState&) const {}
};

// ----------------------------------------------------------------------------- dh

// dS_c [N, width]: K (vocab) contiguous; W_c [width, H]: N (hidden) contiguous.
// hilo: dS is a hi and a lo bf16 plane (columns kBwdChunk apart); the K loop
// runs over the hi plane, then over the lo plane against the same rows of W_c.
struct DhPolicy : SingleRole<false, true> {
    static constexpr bool kKRemap = true;
    static constexpr bool kCtaPair = true;       // 256-token tiles on a CTA pair

    const int64_t* targets;
    const uint8_t* mask;
    const float* grad;
    const __nv_bfloat16* weight;   // [V][H]
    float* dh_acc;                 // [N][H]
    __nv_bfloat16* dh;             // [N][H]
    const float* ycoef;            // [N] 1 - p_y, from the dS GEMM
    const int* dom;                // [N] dominant non-target class or -1, from the dS GEMM
    const float* dcoef;            // [N] its fp32 coefficient
    int64_t y_off;                 // global id of this weight block's first row
    int V_global;                  // vocabulary size (target validity)
    RowMap rm;                     // compaction of a masked batch (dh_acc rows are compacted)
    float* dh_out32;               // round_last false: fp32 partial of dh by token [N][H]
    int N, V, H, c0, num_m, num_n, kblocks;
    bool first, last;
    bool round_last;               // false: the last chunk writes dh_out32, unrounded
    bool terms;                    // false: no fp32 target terms (no targets)
    bool hilo;                     // dS as hi and lo planes: K runs over both
    float temp;

    __device__ int num_units() const { return rm.tiles(N) * num_n; }
    __device__ int k_blocks(int) const { return hilo ? 2 * kblocks : kblocks; }
    __device__ void k_remap(int kb, int nkb, int&, int& a_k, int&, int& b_k) const {
        if (hilo && kb >= nkb / 2) {
            const int j = kb - nkb / 2;
            a_k = kBwdChunk + j * 64;
            b_k = c0 + j * 64;
        }
    }
    __device__ int tiles_in_unit(int) const { return 1; }
    // unit -> (token tile m, hidden tile n) in row order.  (Grouping 8 hidden tiles
    // cut the modelled DRAM reads by a fifth but measured 1% slower on GB300.)
    __device__ void unit(int u, int& m, int& n) const {
        m = u / num_n;
        n = u - m * num_n;
    }
    __device__ void coords(int u, int, int& a_mn, int& a_k, int& b_mn, int& b_k) const {
        int m, n;
        unit(u, m, n);
        a_mn = m * kUnitM;
        a_k = 0;
        b_mn = n * kTileV;
        b_k = c0;
    }

    struct EpiState {
        float coef, coef_dom;
        int64_t y;                 // target row inside this weight block
        int dom;
        int t;                     // the row's token (N past the compacted rows)
        bool live, tgt;            // tgt: the row's target term belongs to this block
    };

    __device__ void epi_begin(int u, int row, EpiState& st) const {
        int m, n;
        unit(u, m, n);
        const int i = m * kUnitM + row;
        const int t = i < rm.count(N) ? rm.token(i) : N;
        st.t = t;
        // the fp32 terms, added once, in the last chunk's epilogue: (g / T)(1 - p_y) W[y]
        // and, for a dominant non-target class a, dcoef W[a]
        if (terms) {
            st.live = row_live(targets, mask, t, N, V_global, st.y);
            st.y -= y_off;
            st.tgt = st.live && last && st.y >= 0 && st.y < V;
            const float gt = (st.live && last) ? __fdiv_rn(grad[t], temp) : 0.f;
            st.coef = st.tgt ? gt * ycoef[t] : 0.f;
        } else {
            st.live = t < N && (mask == nullptr || mask[t] != 0);
            st.y = 0;
            st.tgt = false;
            st.coef = 0.f;
        }
        st.dom = (st.live && last) ? dom[t] : -1;
        st.coef_dom = st.dom >= 0 ? dcoef[t] : 0.f;
    }

    __device__ void epi_tile(int u, int, int row, uint32_t taddr, EpiState& st) const {
        int m, n;
        unit(u, m, n);
        const int ri = m * kUnitM + row;         // dh_acc row (compacted row)
        const int t = st.t;                      // its token
#pragma unroll 1
        for (int cc = 0; cc < kTileV / 32; ++cc) {
            uint32_t r[32];
            tmem_load_32(taddr + cc * 32, r);
            const int col = n * kTileV + cc * 32;
            if (t >= N || col >= H) continue;    // also the rows past the compacted ones
            float x[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]);
            float* acc = dh_acc + static_cast<size_t>(ri) * H + col;
            if (!first) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 pv = reinterpret_cast<const float4*>(acc)[i];
                    x[4 * i] = pv.x + x[4 * i];
                    x[4 * i + 1] = pv.y + x[4 * i + 1];
                    x[4 * i + 2] = pv.z + x[4 * i + 2];
                    x[4 * i + 3] = pv.w + x[4 * i + 3];
                }
            }
            if (!last) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    reinterpret_cast<float4*>(acc)[i] =
                        make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
                continue;
            }
            if (st.live) {
                if (st.tgt) {
                    const uint4* wr = reinterpret_cast<const uint4*>(
                        weight + static_cast<size_t>(st.y) * H + col);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float wv[8];
                        bf16x8_to_f32(wr[i], wv);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            x[8 * i + j] = fmaf(st.coef, wv[j], x[8 * i + j]);
                    }
                }
                if (st.dom >= 0) {
                    const uint4* wa = reinterpret_cast<const uint4*>(
                        weight + static_cast<size_t>(st.dom) * H + col);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float wv[8];
                        bf16x8_to_f32(wa[i], wv);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            x[8 * i + j] = fmaf(st.coef_dom, wv[j], x[8 * i + j]);
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) x[j] = 0.f;
            }
            if (!round_last) {             // a vocab block's fp32 partial of dh
                float* out = dh_out32 + static_cast<size_t>(t) * H + col;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    reinterpret_cast<float4*>(out)[q] =
                        make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
                continue;
            }
            uint4* dst = reinterpret_cast<uint4*>(dh + static_cast<size_t>(t) * H + col);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(pack_bf16x2(x[8 * i], x[8 * i + 1]),
                                    pack_bf16x2(x[8 * i + 2], x[8 * i + 3]),
                                    pack_bf16x2(x[8 * i + 4], x[8 * i + 5]),
                                    pack_bf16x2(x[8 * i + 6], x[8 * i + 7]));
        }
    }

    __device__ void epi_end(int, int, EpiState&) const {}
};

// ----------------------------------------------------------------------------- dW

// dS_c^T: vocab (M) contiguous, tokens along K; h: hidden (N) contiguous.
// hilo: the K loop runs over the tokens of the hi plane of dS, then over the
// same tokens of the lo plane (kBwdChunk columns further on), against h twice.
struct DwPolicy : SingleRole<true, true> {
    static constexpr bool kKRemap = true;
    static constexpr bool kCtaPair = true;       // 256-vocab-row tiles on a CTA pair

    const float* grad;
    const __nv_bfloat16* hidden;   // [N][H]
    __nv_bfloat16* dw;             // [V][H]
    const int* sorted_y;           // [N] ascending; V marks rows without a target term
    const int* sorted_t;           // [N]
    const float* ycoef;            // [N] 1 - p_y, from the dS GEMM
    const int* sorted_dy;          // [N] dominant class of this chunk ascending, V elsewhere
    const int* sorted_dt;          // [N]
    const int* dom_flag;           // 0: no dominant class in this chunk (the list was not built)
    const float* dcoef;            // [N] fp32 coefficient of each token's dominant class
    float* dw_out32;               // non-null: dW rows go here in fp32, unrounded [V][H]
    RowMap rm;                     // compaction: K runs over the compacted rows only
    int N, H, c0, width, num_m, num_n, kblocks;
    float temp;
    bool terms;                    // false: no fp32 target terms (no targets)
    bool hilo;                     // dS as hi and lo planes: K runs over both

    __device__ int num_units() const { return num_m * num_n; }
    __device__ int k_blocks(int) const {
        const int kb = rm.n_rows != nullptr ? (max(*rm.n_rows, 1) + 63) / 64 : kblocks;
        return hilo ? 2 * kb : kb;
    }
    __device__ void k_remap(int kb, int nkb, int& a_mn, int& a_k, int&, int& b_k) const {
        if (hilo && kb >= nkb / 2) {
            const int j = kb - nkb / 2;
            a_mn += kBwdChunk;
            a_k = j * 64;
            b_k = j * 64;
        }
    }
    __device__ int tiles_in_unit(int) const { return 1; }
    // unit -> (vocab tile m of the chunk, hidden tile n), hidden tiles grouped
    __device__ void unit(int u, int& m, int& n) const {
        grouped_unit(u, num_n, num_m, kRasterHiddenTiles, n, m);
    }
    __device__ void coords(int u, int, int& a_mn, int& a_k, int& b_mn, int& b_k) const {
        int m, n;
        unit(u, m, n);
        a_mn = m * kUnitM;
        a_k = 0;
        b_mn = n * kTileV;
        b_k = 0;
    }

    struct EpiState {
        int lo, hi, dlo, dhi, v;
        bool valid;
    };

    // [lo, hi): the entries of an ascending list equal to v
    __device__ static void equal_range(const int* keys, int n, int v, int& lo, int& hi) {
        int a = 0, b = n;
        while (a < b) {
            const int mid = (a + b) >> 1;
            if (keys[mid] < v) a = mid + 1; else b = mid;
        }
        int e = a;
        while (e < n && keys[e] == v) ++e;
        lo = a;
        hi = e;
    }

    __device__ void epi_begin(int u, int row, EpiState& st) const {
        int m, n;
        unit(u, m, n);
        const int vl = m * kUnitM + row;
        st.valid = vl < width;
        st.v = c0 + vl;
        st.lo = st.hi = st.dlo = st.dhi = 0;
        if (!st.valid) return;
        if (terms) equal_range(sorted_y, N, st.v, st.lo, st.hi);
        if (*dom_flag != 0) equal_range(sorted_dy, N, st.v, st.dlo, st.dhi);
    }

    __device__ void epi_tile(int u, int, int, uint32_t taddr, EpiState& st) const {
        int m, n;
        unit(u, m, n);
#pragma unroll 1
        for (int cc = 0; cc < kTileV / 32; ++cc) {
            uint32_t r[32];
            tmem_load_32(taddr + cc * 32, r);
            const int col = n * kTileV + cc * 32;
            if (!st.valid || col >= H) continue;
            float x[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]);
            for (int i = st.lo; i < st.hi; ++i) {
                const int t = sorted_t[i];
                const float coef = __fdiv_rn(grad[t], temp) * ycoef[t];
                const uint4* hr = reinterpret_cast<const uint4*>(
                    hidden + static_cast<size_t>(t) * H + col);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float hv[8];
                    bf16x8_to_f32(hr[q], hv);
#pragma unroll
                    for (int j = 0; j < 8; ++j) x[8 * q + j] = fmaf(coef, hv[j], x[8 * q + j]);
                }
            }
            // tokens whose dominant non-target class is v: dcoef_t h_t, ascending t
            for (int i = st.dlo; i < st.dhi; ++i) {
                const int t = sorted_dt[i];
                const float coef = dcoef[t];
                const uint4* hr = reinterpret_cast<const uint4*>(
                    hidden + static_cast<size_t>(t) * H + col);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float hv[8];
                    bf16x8_to_f32(hr[q], hv);
#pragma unroll
                    for (int j = 0; j < 8; ++j) x[8 * q + j] = fmaf(coef, hv[j], x[8 * q + j]);
                }
            }
            if (dw_out32 != nullptr) {     // a data-parallel rank's unrounded partial
                float4* out = reinterpret_cast<float4*>(dw_out32 + static_cast<size_t>(st.v) * H +
                                                        col);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    out[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
                continue;
            }
            uint4* dst = reinterpret_cast<uint4*>(dw + static_cast<size_t>(st.v) * H + col);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(pack_bf16x2(x[8 * i], x[8 * i + 1]),
                                    pack_bf16x2(x[8 * i + 2], x[8 * i + 3]),
                                    pack_bf16x2(x[8 * i + 4], x[8 * i + 5]),
                                    pack_bf16x2(x[8 * i + 6], x[8 * i + 7]));
        }
    }

    __device__ void epi_end(int, int, EpiState&) const {}
};

// ----------------------------------------------------------------------------- target list

constexpr int kSortTile = kTargetSortTile;  // keys per tile (shared memory: 16 KB)
constexpr int kSortThreads = 1024;
constexpr int kPlaceThreads = 256;
constexpr uint64_t kPadKey = ~0ull;         // above every real key

// Batcher's bitonic network over the block's tile of keys in shared memory:
// merge sorted runs of `size`, comparing at distance `d`.
__device__ __forceinline__ void bitonic_sort_tile(uint64_t* key) {
    for (int size = 2; size <= kSortTile; size <<= 1) {
        for (int d = size >> 1; d > 0; d >>= 1) {
            for (int i = threadIdx.x; i < kSortTile; i += kSortThreads) {
                const int j = i ^ d;
                if (j > i) {
                    const bool ascending = (i & size) == 0;
                    const uint64_t a = key[i], b = key[j];
                    if ((a > b) == ascending) {
                        key[i] = b;
                        key[j] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
}

// Keys (target, token) of the dW target terms; also resets dom[] to "no dominant class"
// and the chunks' flags to "no dominant class in this chunk".
__global__ void __launch_bounds__(kSortThreads)
    target_tile_sort_kernel(const int64_t* __restrict__ targets, const uint8_t* __restrict__ mask,
                            int N, int V, int64_t y_off, int V_global,
                            uint64_t* __restrict__ tiles, int* __restrict__ dom,
                            int* __restrict__ dom_flags, int num_chunks, uint32_t* err) {
    __shared__ uint64_t key[kSortTile];
    const int base = blockIdx.x * kSortTile;
    if (blockIdx.x == 0)
        for (int c = threadIdx.x; c < num_chunks; c += kSortThreads) dom_flags[c] = 0;
    for (int i = threadIdx.x; i < kSortTile; i += kSortThreads) {
        const int t = base + i;
        uint64_t k = kPadKey;
        if (t < N) {
            int y = V;                          // V: no target term in this block
            if (mask == nullptr || mask[t] != 0) {
                const int64_t yt = targets[t];
                if (yt >= 0 && yt < V_global) {
                    const int64_t yl = yt - y_off;
                    if (yl >= 0 && yl < V) y = static_cast<int>(yl);
                } else if (err != nullptr) {
                    atomicOr(err, RLK_DEVERR_TARGET_RANGE);
                }
            }
            k = (static_cast<uint64_t>(y) << 32) | static_cast<uint32_t>(t);
            dom[t] = -1;
        }
        key[i] = k;
    }
    __syncthreads();
    bitonic_sort_tile(key);
    for (int i = threadIdx.x; i < kSortTile; i += kSortThreads) tiles[base + i] = key[i];
}

// Keys (dominant class, token) of the tokens whose dominant non-target class lies in
// [lo, hi) (one vocab chunk); V for every other token.  Nothing to do when the dS
// GEMM found no dominant class in the chunk (its flag is 0); dW then reads no list.
__global__ void __launch_bounds__(kSortThreads)
    dom_tile_sort_kernel(const int* __restrict__ dom, int N, int V, int lo, int hi,
                         const int* __restrict__ flag, uint64_t* __restrict__ tiles) {
    if (*flag == 0) return;
    __shared__ uint64_t key[kSortTile];
    const int base = blockIdx.x * kSortTile;
    for (int i = threadIdx.x; i < kSortTile; i += kSortThreads) {
        const int t = base + i;
        uint64_t k = kPadKey;
        if (t < N) {
            const int a = dom[t];
            const int c = (a >= lo && a < hi) ? a : V;
            k = (static_cast<uint64_t>(c) << 32) | static_cast<uint32_t>(t);
        }
        key[i] = k;
    }
    __syncthreads();
    bitonic_sort_tile(key);
    for (int i = threadIdx.x; i < kSortTile; i += kSortThreads) tiles[base + i] = key[i];
}

__global__ void __launch_bounds__(kPlaceThreads)
    target_place_kernel(const uint64_t* __restrict__ tiles, int num_tiles,
                        const int* __restrict__ flag, int* __restrict__ sorted_y,
                        int* __restrict__ sorted_t) {
    if (flag != nullptr && *flag == 0) return;    // an empty dominant-class list
    const int e = blockIdx.x * kPlaceThreads + threadIdx.x;
    if (e >= num_tiles * kSortTile) return;
    const uint64_t k = tiles[e];
    if (k == kPadKey) return;
    const int own = e / kSortTile;
    int rank = e - own * kSortTile;
    for (int b = 0; b < num_tiles; ++b) {
        if (b == own) continue;
        const uint64_t* tile = tiles + static_cast<size_t>(b) * kSortTile;
        int lo = 0, hi = kSortTile;              // first index whose key is not below k
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (tile[mid] < k) lo = mid + 1; else hi = mid;
        }
        rank += lo;
    }
    sorted_y[rank] = static_cast<int>(k >> 32);
    sorted_t[rank] = static_cast<int>(k & 0xffffffffu);
}

static cudaError_t place_sorted(const uint64_t* tiles, int N, const int* flag, int* sorted_key,
                                int* sorted_t, cudaStream_t stream) {
    const int num_tiles = (N + kSortTile - 1) / kSortTile;
    const int total = num_tiles * kSortTile;
    target_place_kernel<<<(total + kPlaceThreads - 1) / kPlaceThreads, kPlaceThreads, 0, stream>>>(
        tiles, num_tiles, flag, sorted_key, sorted_t);
    return cudaGetLastError();
}

cudaError_t launch_target_sort(const int64_t* targets, const uint8_t* mask, int N, int V,
                               int64_t y_off, int V_global, uint64_t* tiles, int* sorted_y,
                               int* sorted_t, int* dom, int* dom_flags, int num_chunks,
                               uint32_t* err, cudaStream_t stream) {
    const int num_tiles = (N + kSortTile - 1) / kSortTile;
    target_tile_sort_kernel<<<num_tiles, kSortThreads, 0, stream>>>(
        targets, mask, N, V, y_off, V_global, tiles, dom, dom_flags, num_chunks, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return place_sorted(tiles, N, nullptr, sorted_y, sorted_t, stream);
}

static cudaError_t launch_dom_sort(const int* dom, int N, int V, int lo, int hi, const int* flag,
                                   uint64_t* tiles, int* sorted_dy, int* sorted_dt,
                                   cudaStream_t stream) {
    const int num_tiles = (N + kSortTile - 1) / kSortTile;
    dom_tile_sort_kernel<<<num_tiles, kSortThreads, 0, stream>>>(dom, N, V, lo, hi, flag, tiles);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return place_sorted(tiles, N, flag, sorted_dy, sorted_dt, stream);
}

// ----------------------------------------------------------------------------- launch

template <class P>
static cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const P& p, int units,
                               int num_sms, uint32_t* err, cudaStream_t stream,
                               unsigned pdl = 0) {
    return launch_persistent(TwoMaps{a, b}, p, units, num_sms, err, stream, pdl);
}

template <bool ENT>
static cudaError_t launch_ds(const BwdStepMaps& maps, const BwdStep& st, int c0, int width,
                             int num_sms, uint32_t* err, cudaStream_t stream) {
    DsPolicyT<ENT> ps;
    ps.targets = st.targets;
    ps.mask = st.mask;
    ps.grad = st.grad;
    ps.grad_ent = st.grad_ent;
    ps.ent = st.ent;
    ps.lse = st.lse;
    ps.ds = static_cast<__nv_bfloat16*>(st.ds);
    ps.ycoef = st.ycoef;
    ps.dom = st.dom;
    ps.dcoef = st.dcoef;
    ps.y_off = st.y_off;
    ps.V_global = st.V_global;
    ps.rm = RowMap{st.rows, st.n_rows};
    ps.dom_flag = st.dom_flags + st.chunk;
    ps.N = st.N;
    ps.V = st.V;
    ps.c0 = c0;
    ps.num_m = (st.N + kUnitM - 1) / kUnitM;
    ps.num_n = (width + kTileV - 1) / kTileV;
    ps.kblocks = st.H / 64;
    ps.k = st.k;
    ps.temp = st.temp;
    return launch_gemm(maps.h_kmajor, maps.w_kmajor_pair, ps, ps.num_m * ps.num_n, num_sms, err,
                       stream);
}

cudaError_t launch_bwd_step(const BwdStepMaps& maps, const BwdStep& st, int num_sms, uint32_t* err,
                            cudaStream_t stream) {
    const int N = st.N, H = st.H, V = st.V;
    const int c0 = st.chunk * kBwdChunk;
    const int width = (V - c0) < kBwdChunk ? (V - c0) : kBwdChunk;
    if (st.role == kRoleDs && st.kl) {
        DsKlPolicy ps;
        ps.mask = st.mask;
        ps.grad = st.grad;
        ps.grad_rev = st.grad_rev;
        ps.lse = st.lse;
        ps.lse_ref = st.lse_ref;
        ps.kl = st.kl_val;
        ps.ds = static_cast<__nv_bfloat16*>(st.ds);
        ps.dom = st.dom;
        ps.dcoef = st.dcoef;
        ps.dom_flag = st.dom_flags + st.chunk;
        ps.N = N;
        ps.V = V;
        ps.c0 = c0;
        ps.num_m = (N + kUnitM - 1) / kUnitM;
        ps.num_n = (width + kTileV - 1) / kTileV;
        ps.kblocks = H / 64;
        ps.kblocks_r = st.H_ref / 64;
        ps.k = st.k;
        ps.kr = st.k_ref;
        ps.temp = st.temp;
        const long long units = static_cast<long long>(ps.num_m) * ps.num_n;
        const cudaError_t e = launch_persistent<DsKlPolicy>(
            DsKlMaps{maps.h_kmajor, maps.w_kmajor, maps.hr_kmajor, maps.wr_kmajor, maps.ds_store},
            ps, units, num_sms, err, stream);
        if (e != cudaSuccess) return e;
        return launch_dom_sort(st.dom, N, V, c0, c0 + width, st.dom_flags + st.chunk, st.tiles,
                               st.sorted_dy, st.sorted_dt, stream);
    }
    if (st.role == kRoleDs) {
        const cudaError_t e =
            st.grad_ent != nullptr ? launch_ds<true>(maps, st, c0, width, num_sms, err, stream)
                                   : launch_ds<false>(maps, st, c0, width, num_sms, err, stream);
        if (e != cudaSuccess) return e;
        // the tokens whose dominant non-target class the dS GEMM found in this chunk
        return launch_dom_sort(st.dom, N, V, c0, c0 + width, st.dom_flags + st.chunk, st.tiles,
                               st.sorted_dy, st.sorted_dt, stream);
    }
    if (st.role == kRoleDh) {
        DhPolicy pd;
        pd.targets = st.targets;
        pd.mask = st.mask;
        pd.grad = st.grad;
        pd.weight = static_cast<const __nv_bfloat16*>(st.weight);
        pd.dh_acc = st.dh_acc;
        pd.dh = static_cast<__nv_bfloat16*>(st.dhidden);
        pd.ycoef = st.ycoef;
        pd.dom = st.dom;
        pd.dcoef = st.dcoef;
        pd.y_off = st.y_off;
        pd.V_global = st.V_global;
        pd.round_last = st.round_last;
        pd.rm = RowMap{st.rows, st.n_rows};
        pd.dh_out32 = st.dh_out32;
        pd.N = N;
        pd.V = V;
        pd.H = H;
        pd.c0 = c0;
        pd.num_m = (N + kUnitM - 1) / kUnitM;
        pd.num_n = (H + kTileV - 1) / kTileV;
        pd.kblocks = (width + 63) / 64;
        pd.first = st.chunk == 0;
        pd.last = st.chunk == st.num_chunks - 1;
        pd.temp = st.temp;
        pd.terms = !st.kl;
        pd.hilo = st.hilo;
        // the dW GEMM that follows overlaps this one's last wave (with 6.7 waves of dh
        // units at N = 8192, a quarter of the CTA pairs would otherwise idle for a unit)
        return launch_gemm(maps.ds_kmajor, maps.w_mnmajor, pd, pd.num_m * pd.num_n, num_sms, err,
                           stream, kPdlTrigger);
    }
    DwPolicy pw;
    pw.grad = st.grad;
    pw.hidden = static_cast<const __nv_bfloat16*>(st.hidden);
    pw.dw = static_cast<__nv_bfloat16*>(st.dweight);
    pw.sorted_y = st.sorted_y;
    pw.sorted_t = st.sorted_t;
    pw.ycoef = st.ycoef;
    pw.sorted_dy = st.sorted_dy;
    pw.sorted_dt = st.sorted_dt;
    pw.dom_flag = st.dom_flags + st.chunk;
    pw.dcoef = st.dcoef;
    pw.dw_out32 = st.dw_out32;
    pw.rm = RowMap{st.rows, st.n_rows};
    pw.N = N;
    pw.H = H;
    pw.c0 = c0;
    pw.width = width;
    pw.num_m = (width + kUnitM - 1) / kUnitM;
    pw.num_n = (H + kTileV - 1) / kTileV;
    pw.kblocks = (N + 63) / 64;
    pw.temp = st.temp;
    pw.terms = !st.kl;
    pw.hilo = st.hilo;
    // dW reads dS, h and the target lists, all complete before the dh GEMM started, and
    // writes only dW, which the dh GEMM does not touch
    return launch_gemm(maps.ds_mnmajor, maps.h_mnmajor, pw, pw.num_m * pw.num_n, num_sms, err,
                       stream, kPdlOverlap);
}

// ----------------------------------------------------------------------------- dh merge

// out = bf16( sum_r partials[r] ), r ascending, fp32 sums; four elements a thread.
// Serves the vocab-sharded backward's dh partials and the data-parallel ranks'
// dW partials alike.
__global__ void dh_merge_kernel(const float4* __restrict__ partials, int64_t num_parts,
                                int64_t n4, uint2* __restrict__ dh) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n4) return;
    float4 a = partials[i];
    for (int64_t r = 1; r < num_parts; ++r) {
        const float4 b = partials[r * n4 + i];
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
    }
    dh[i] = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
}

cudaError_t launch_dh_merge(const float* partials, int64_t num_parts, int64_t N, int64_t H,
                            void* dhidden, cudaStream_t stream) {
    const int64_t n4 = N * H / 4;                  // H is a multiple of 64
    if (n4 == 0) return cudaSuccess;
    dh_merge_kernel<<<static_cast<unsigned>((n4 + 255) / 256), 256, 0, stream>>>(
        reinterpret_cast<const float4*>(partials), num_parts, n4, static_cast<uint2*>(dhidden));
    return cudaGetLastError();
}

}  // namespace rlk
