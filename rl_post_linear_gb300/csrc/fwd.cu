// fwd.cu -- forward of the fused linear selected-token log-prob.
//
// "RL-Kernel Roadmap (2026)", P0.2 Typical Fused Operators: the forward
// streams vocab blocks with an online softmax and never lands the [N,V]
// logits.  "RL-Kernel integration roadmap for vime", linear_logp section:
// here each (row, vocab chunk) leaves a running maximum and a scaled sum of
// exponentials, the row's target logit is kept from the same accumulator, and
// a separate launch merges the per-chunk pairs in one fixed order before the
// single fp32 result is formed.
//
// Kernel 1 (gemm_persistent_kernel<FwdPolicy>): a work unit is one 256-row
// token tile, computed by a CTA pair (128 rows in each CTA's TMEM), times one
// vocab chunk of kFwdTilesPerChunk 256-column tiles.  For every tile the
// tensor cores form S = h W^T in TMEM (fp32, K = H in ascending 16-wide
// steps); one epilogue thread owns one token row and folds
// the tile's 256 logits, 32 at a time and in ascending column order, into
// the row's running (max m, sum s) with
//     m' = max(m, max_j S_j),  s' = s 2^((m - m') k) + sum_j 2^((S_j - m') k),
// k = log2(e)/T.  Columns >= V are excluded.  The target logit S[t, y_t] is
// taken from the same accumulator.  At the end of the unit it writes the
// chunk's partial (m, s), and the target logit if the chunk holds y_t.
//
// Kernel 2 (fwd_merge_kernel): eight threads per row merge the partials of the
// chunks, each the chunks c = g (mod 8) in ascending order, then one of them
// the eight groups in ascending order, each level as
//     M = max m,  sigma = sum s 2^((m - M) k);
// then lse2 = M k + log2(sigma),  logp = (S_y k - lse2) ln 2,  lse = lse2 ln 2.
// Inactive rows get logp = lse = 0; an active row with an out-of-range target
// gets logp = NaN and raises RLK_DEVERR_TARGET_RANGE.
//
// Batch invariance: a row's arithmetic is a fixed sequence -- the same K
// order, the same 32-column slices, the same chunk boundaries (functions of
// V only) and the same merge order -- whatever the row's tile, lane, batch or
// the number of SMs.  No atomics touch any float.
#include <cmath>

#include "gemm.cuh"

namespace rlk {


// Stand-in for the logits of columns past V: far below any logit, so that
// 2^((x - m) k) underflows to exactly 0, and finite, so that 0 * x stays 0.
constexpr float kMaskedLogit = -3.0e38f;

// ENT adds the running sum a = sum_j 2^((S_j - m) k) S_j per row, from which
// the merge forms E[S] = a / s and the entropy lse - E[S]/T.
template <bool ENT>
struct FwdPolicyT : SingleRole<false, false> {   // h [N,H] and W [V,H]: K-major
    static constexpr bool kCtaPair = true;       // 256-token tiles on a CTA pair

    const int64_t* targets;
    const uint8_t* mask;
    float2* partials;     // [num_chunks][N]
    float* partials_a;    // [num_chunks][N] (ENT only)
    float* s_target;      // [N]
    const int* rows;      // compacted row -> token (nullptr: rows are tokens)
    const int* n_rows;    // number of compacted rows, on the device (nullptr: N)
    int64_t vocab_start;  // global id of this weight block's first row
    int N, V, num_m, num_vt, num_chunks, kblocks;   // V: rows of this weight block
    float k;              // log2(e) / T

    __device__ int valid_rows() const { return n_rows != nullptr ? *n_rows : N; }
    __device__ int token_tiles() const {
        return n_rows != nullptr ? (*n_rows + kUnitM - 1) / kUnitM : num_m;
    }

    __device__ int num_units() const { return token_tiles() * num_chunks; }
    __device__ int k_blocks(int) const { return kblocks; }
    // unit -> (token tile m, vocab chunk c), token tiles grouped kRasterTokenRows rows at a time
    __device__ void unit(int u, int& m, int& c) const {
        grouped_unit(u, token_tiles(), num_chunks, kRasterTokenRows / kUnitM, m, c);
    }
    __device__ int tiles_in_unit(int u) const {
        int m, c;
        unit(u, m, c);
        return min(kFwdTilesPerChunk, num_vt - c * kFwdTilesPerChunk);
    }
    __device__ void coords(int u, int q, int& a_mn, int& a_k, int& b_mn, int& b_k) const {
        int m, c;
        unit(u, m, c);
        a_mn = m * kUnitM;
        a_k = 0;
        b_mn = (c * kFwdTilesPerChunk + q) * kTileV;
        b_k = 0;
    }

    struct EpiState {
        float m, s, a, sy;
        int64_t y;
        bool found;
    };

    __device__ void epi_begin(int u, int row, EpiState& st) const {
        int m, c;
        unit(u, m, c);
        const int i = m * kUnitM + row;
        st.m = -INFINITY;
        st.s = 0.f;
        st.a = 0.f;
        st.sy = 0.f;
        st.found = false;
        st.y = -1;
        if (i < valid_rows()) {
            const int t = rows != nullptr ? rows[i] : i;
            if (mask == nullptr || mask[t] != 0) st.y = targets[t];
        }
    }

    __device__ void epi_tile(int u, int q, int row, uint32_t taddr, EpiState& st) const {
        int m, c;
        unit(u, m, c);
        const int v0 = (c * kFwdTilesPerChunk + q) * kTileV;
#pragma unroll 1
        for (int cc = 0; cc < kTileV / 32; ++cc) {
            const int vb = v0 + cc * 32;
            if (vb >= V) break;                       // same for the whole warp
            uint32_t r[32];
            tmem_load_32(taddr + cc * 32, r);
            float x[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]);
            const int nv = V - vb;
            if (nv < 32) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j >= nv) x[j] = kMaskedLogit;
            }
            const int64_t dy = st.y - vocab_start - vb;
            if (dy >= 0 && dy < 32) {
                st.sy = select32(x, static_cast<int>(dy));
                st.found = true;
            }
            const float cm = max32(x);
            const float nm = fmaxf(st.m, cm);
            const float rescale = ex2_approx((st.m - nm) * k);
            const float nmk = nm * k;                 // each exponent: one fma, x k - m k
            float acc = st.s * rescale;
            if constexpr (ENT) {
                float aa = st.a * rescale;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float e = ex2_approx(fmaf(x[j], k, -nmk));
                    acc += e;
                    aa = fmaf(e, x[j], aa);
                }
                st.a = aa;
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) acc += ex2_approx(fmaf(x[j], k, -nmk));
            }
            st.s = acc;
            st.m = nm;
        }
    }

    __device__ void epi_end(int u, int row, EpiState& st) const {
        int m, c;
        unit(u, m, c);
        const int i = m * kUnitM + row;          // compacted row (the token when not compacted)
        if (i >= valid_rows()) return;
        partials[static_cast<size_t>(c) * N + i] = make_float2(st.m, st.s);
        if constexpr (ENT) partials_a[static_cast<size_t>(c) * N + i] = st.a;
        if (st.found) s_target[i] = st.sy;
    }
};

// The merge: kMergeRows rows per block, each row's chunks dealt to kMergeGroups
// threads (chunk c to group c mod kMergeGroups, so consecutive rows of a group
// read consecutive addresses).  Each group merges its chunks in ascending order
// (its max, then the rescaled sums); thread group 0 then merges the groups in
// ascending order the same way.  A fixed two-level order, a function of the row
// and of V only: batch invariant, no atomics.
constexpr int kMergeRows = 32;
constexpr int kMergeGroups = 8;

__global__ void __launch_bounds__(kMergeRows * kMergeGroups)
    fwd_merge_kernel(const float2* __restrict__ partials, const float* __restrict__ partials_a,
                     const float* __restrict__ s_target, const int* __restrict__ pos_of,
                     const int64_t* __restrict__ targets, const uint8_t* __restrict__ mask,
                     int N, int V, int num_chunks, float k, float* __restrict__ logp,
                     float* __restrict__ lse, float* __restrict__ entropy, uint32_t* err) {
    __shared__ float s_m[kMergeGroups][kMergeRows];
    __shared__ float s_s[kMergeGroups][kMergeRows];
    __shared__ float s_a[kMergeGroups][kMergeRows];
    const int r = threadIdx.x % kMergeRows;
    const int g = threadIdx.x / kMergeRows;
    const int t = blockIdx.x * kMergeRows + r;
    const bool live = t < N && (mask == nullptr || mask[t] != 0);
    const int i = !live ? 0 : (pos_of != nullptr ? pos_of[t] : t);   // the token's partials row
    float m = -INFINITY, sigma = 0.f, a = 0.f;
    if (live) {
        for (int c = g; c < num_chunks; c += kMergeGroups)
            m = fmaxf(m, partials[static_cast<size_t>(c) * N + i].x);
        for (int c = g; c < num_chunks; c += kMergeGroups) {
            const float2 pc = partials[static_cast<size_t>(c) * N + i];
            const float wgt = ex2_approx((pc.x - m) * k);
            sigma += pc.y * wgt;
            if (entropy != nullptr) a += partials_a[static_cast<size_t>(c) * N + i] * wgt;
        }
    }
    s_m[g][r] = m;
    s_s[g][r] = sigma;
    s_a[g][r] = a;
    __syncthreads();
    if (g != 0 || t >= N) return;
    if (!live) {
        logp[t] = 0.f;
        if (lse != nullptr) lse[t] = 0.f;
        if (entropy != nullptr) entropy[t] = 0.f;
        return;
    }
    float mm = -INFINITY;
#pragma unroll
    for (int q = 0; q < kMergeGroups; ++q) mm = fmaxf(mm, s_m[q][r]);
    float sg = 0.f, ag = 0.f;
#pragma unroll
    for (int q = 0; q < kMergeGroups; ++q) {
        const float wgt = ex2_approx((s_m[q][r] - mm) * k);   // 0 for a group without chunks
        sg += s_s[q][r] * wgt;
        ag += s_a[q][r] * wgt;
    }
    const float lse2 = mm * k + lg2_approx(sg);
    constexpr float kLn2 = 0.693147180559945309f;
    if (lse != nullptr) lse[t] = lse2 * kLn2;
    if (entropy != nullptr) entropy[t] = (lse2 - (ag / sg) * k) * kLn2;
    const int64_t y = targets[t];
    if (y < 0 || y >= V) {
        logp[t] = __int_as_float(0x7fc00000);
        if (err != nullptr) atomicOr(err, RLK_DEVERR_TARGET_RANGE);
        return;
    }
    logp[t] = (s_target[i] * k - lse2) * kLn2;
}

template <bool ENT>
static cudaError_t launch_partials_t(const CUtensorMap& map_h, const CUtensorMap& map_w,
                                     const int64_t* targets, const uint8_t* mask, int N, int H,
                                     int V_local, int64_t vocab_start, float k, float2* partials,
                                     float* partials_a, float* s_target, const int* rows,
                                     const int* n_rows, uint32_t* err, int num_sms,
                                     cudaStream_t stream) {
    FwdPolicyT<ENT> p;
    p.targets = targets;
    p.mask = mask;
    p.partials = partials;
    p.partials_a = partials_a;
    p.s_target = s_target;
    p.rows = rows;
    p.n_rows = n_rows;
    p.vocab_start = vocab_start;
    p.N = N;
    p.V = V_local;
    p.num_m = (N + kUnitM - 1) / kUnitM;
    p.num_vt = (V_local + kTileV - 1) / kTileV;
    p.num_chunks = (p.num_vt + kFwdTilesPerChunk - 1) / kFwdTilesPerChunk;
    p.kblocks = H / 64;
    p.k = k;
    const long long units = static_cast<long long>(p.num_m) * p.num_chunks;
    return launch_persistent(TwoMaps{map_h, map_w}, p, units, num_sms, err, stream);
}

cudaError_t launch_fwd_partials(const CUtensorMap& map_h, const CUtensorMap& map_w,
                                const int64_t* targets, const uint8_t* mask, int N, int H,
                                int V_local, int64_t vocab_start, float k, float2* partials,
                                float* s_target, uint32_t* err, int num_sms, cudaStream_t stream) {
    return launch_partials_t<false>(map_h, map_w, targets, mask, N, H, V_local, vocab_start, k,
                                    partials, nullptr, s_target, nullptr, nullptr, err, num_sms,
                                    stream);
}

cudaError_t launch_fwd_merge(const float2* partials, int num_chunks, const float* s_target,
                             const int64_t* targets, const uint8_t* mask, int N, int V, float k,
                             float* logp, float* lse, uint32_t* err, cudaStream_t stream) {
    fwd_merge_kernel<<<(N + kMergeRows - 1) / kMergeRows, kMergeRows * kMergeGroups, 0, stream>>>(
        partials, nullptr, s_target, nullptr, targets, mask, N, V, num_chunks, k, logp, lse,
        nullptr, err);
    return cudaGetLastError();
}

cudaError_t launch_fwd(const CUtensorMap& map_h, const CUtensorMap& map_w, const int64_t* targets,
                       const uint8_t* mask, int N, int H, int V, float k, float* logp, float* lse,
                       float* entropy, void* workspace, const int* rows, const int* n_rows,
                       const int* pos_of, uint32_t* err, int num_sms, cudaStream_t stream) {
    FwdLayout lay(N, H, V);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float2* partials = reinterpret_cast<float2*>(ws + lay.partial_off);
    float* partials_a = reinterpret_cast<float*>(ws + lay.partial_a_off);
    float* s_target = reinterpret_cast<float*>(ws + lay.target_off);
    cudaError_t e = entropy != nullptr
        ? launch_partials_t<true>(map_h, map_w, targets, mask, N, H, V, 0, k, partials, partials_a,
                                  s_target, rows, n_rows, err, num_sms, stream)
        : launch_partials_t<false>(map_h, map_w, targets, mask, N, H, V, 0, k, partials, nullptr,
                                   s_target, rows, n_rows, err, num_sms, stream);
    if (e != cudaSuccess) return e;
    fwd_merge_kernel<<<(N + kMergeRows - 1) / kMergeRows, kMergeRows * kMergeGroups, 0, stream>>>(
        partials, entropy != nullptr ? partials_a : nullptr, s_target, pos_of, targets, mask, N, V,
        static_cast<int>(lay.num_chunks), k, logp, lse, entropy, err);
    return cudaGetLastError();
}

}  // namespace rlk
