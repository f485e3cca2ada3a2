// kl.cu -- full-vocabulary KL between the policy head and a reference head.
//
// "RL-Kernel Roadmap (2026)", backlog: chunked full-vocab KL / distillation KL
// fused with lm_head, forward and reverse KL over the whole distribution
// rather than at the sampled token.  "RL-Kernel integration roadmap for vime",
// linear_logp: the same max / sum-exp statistics and explicit merge.
//
// With policy logits S = h W^T (temperature T, k = log2(e)/T) and reference
// logits R = hr Wr^T (temperature Tr, kr = log2(e)/Tr), in log2 units
// d_v = S_v k - R_v kr, and
//   KL(p || q) = ln2 ( E_p[d] - lse2 + lse2r ),
//   KL(q || p) = ln2 ( -E_q[d] + lse2 - lse2r ).
//
// Kernel 1 (gemm_persistent_kernel<KlFwdPolicy>): a work unit is one 128-row
// token tile times one vocab chunk of kFwdTilesPerChunk 256-column tiles, each
// tile computed twice -- policy then reference -- into the two TMEM
// accumulators (the mainloop's paired-tile mode).  One epilogue thread owns a
// row and folds both tiles, 32 columns at a time in ascending order, into
//   (m, s, a)  = running max of S, sum 2^((S - m) k), sum 2^((S - m) k) d
//   (mr, sr, b) = the same for R with weights 2^((R - mr) kr) and values -d
// and takes the target logit S[t, y_t] from the policy accumulator.  Columns
// >= V are excluded.  At the end of a unit it writes the chunk's partials.
// It runs on single CTAs: on CTA pairs it took 7 % fewer cycles but read the
// two heads' weights from DRAM about 2.5 times as often (54 against 22 GB at
// N = 8192), which under the power cap cost more than the cycles saved.  (The
// KL backward's dS GEMM, whose weight traffic does not grow that way, runs on
// pairs.)
//
// Kernel 2 (kl_merge_kernel): one thread per row merges the chunks in
// ascending order (max, then rescaled sums) and forms KL, reverse KL, both
// log-partition functions and, given targets, the policy's selected logp.
// Every step is a fixed function of the row and of V: batch invariant, no
// float atomics.
#include <cmath>

#include "gemm.cuh"

namespace rlk {

namespace {

constexpr float kLn2f = 0.69314718055994531f;

struct KlMaps {
    CUtensorMap h, w;     // policy hidden [N,H] {64,128}, weight [V,H] {64,256}: K-major
    CUtensorMap hr, wr;   // reference hidden [N,Hr], weight [V,Hr]
};

struct KlFwdPolicy {
    using Maps = KlMaps;
    static constexpr bool kPairTiles = true;
    static constexpr bool kKRemap = false;
    static constexpr bool kCtaPair = false;
    static constexpr int kEpiWarps = 8;       // two column halves per row
    static constexpr int kEpiSmemPerWarp = 0;

    const int64_t* targets;   // nullptr: no selected logp
    // partials per (chunk, column half, row): [num_chunks][2][N]
    float2* part_p;           // (m, s) of the policy
    float* part_a;            // sum 2^((S - m) k) d
    float2* part_r;           // (mr, sr) of the reference
    float* part_b;            // sum 2^((R - mr) kr) (-d)
    float* s_target;          // [N]
    int N, V, num_m, num_vt, num_chunks, kblocks, kblocks_r;
    float k, kr;

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

    __device__ int num_units() const { return num_m * num_chunks; }
    __device__ void unit(int u, int& m, int& c) const {
        grouped_unit(u, num_m, num_chunks, (kRasterTokenRows / kTileM), m, c);
    }
    __device__ int tiles_in_unit(int u) const {
        int m, c;
        unit(u, m, c);
        return 2 * min(kFwdTilesPerChunk, num_vt - c * kFwdTilesPerChunk);
    }
    __device__ void coords(int u, int q, int& a_mn, int& a_k, int& b_mn, int& b_k) const {
        int m, c;
        unit(u, m, c);
        a_mn = m * kTileM;
        a_k = 0;
        b_mn = (c * kFwdTilesPerChunk + (q >> 1)) * kTileV;
        b_k = 0;
    }

    struct EpiState {
        float m, s, a, mr, sr, b, sy;
        int64_t y;
        bool found;
    };

    __device__ void epi_begin(int u, int row, int, EpiState& st) const {
        int m, c;
        unit(u, m, c);
        const int t = m * kTileM + row;
        st.m = st.mr = -INFINITY;
        st.s = st.a = st.sr = st.b = st.sy = 0.f;
        st.found = false;
        st.y = (targets != nullptr && t < N) ? targets[t] : -1;
    }

    __device__ void epi_pair(const Maps&, int u, int q, int, int half, uint32_t tp, uint32_t tr,
                             EpiState& st, uint8_t*) const {
        int m, c;
        unit(u, m, c);
        const int v0 = (c * kFwdTilesPerChunk + (q >> 1)) * kTileV;
#pragma unroll 1
        for (int cc = half * (kTileV / 64); cc < (half + 1) * (kTileV / 64); ++cc) {
            const int vb = v0 + cc * 32;
            if (vb >= V) break;                       // same for the whole warp
            uint32_t rp[32], rr[32];
            tmem_load_32x2(tp + cc * 32, rp, tr + cc * 32, rr);
            float x[32], xr[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                x[j] = __uint_as_float(rp[j]);
                xr[j] = __uint_as_float(rr[j]);
            }
            const int nv = V - vb;                    // valid columns in this slice
            const int64_t dy = st.y - vb;
            if (dy >= 0 && dy < 32) {
                st.sy = select32(x, static_cast<int>(dy));
                st.found = true;
            }
            if (nv >= 32)
                fold<true>(x, xr, 32, st);
            else
                fold<false>(x, xr, nv, st);
        }
    }

    // One 32-column slice of both heads into the row's running statistics; FULL
    // (all 32 columns inside the vocabulary, a warp-uniform case) drops the
    // per-column checks.
    template <bool FULL>
    __device__ __forceinline__ void fold(const float (&x)[32], const float (&xr)[32], int nv,
                                         EpiState& st) const {
        float cm = -INFINITY, cmr = -INFINITY;
        if constexpr (FULL) {
            cm = fmaxf(cm, max32(x));
            cmr = fmaxf(cmr, max32(xr));
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (j < nv) {
                    cm = fmaxf(cm, x[j]);
                    cmr = fmaxf(cmr, xr[j]);
                }
            }
        }
        const float nm = fmaxf(st.m, cm), nmr = fmaxf(st.mr, cmr);
        const float sc = ex2_approx((st.m - nm) * k), scr = ex2_approx((st.mr - nmr) * kr);
        const float nmk = __fmul_rn(nm, k), nmrk = __fmul_rn(nmr, kr);
        float s = st.s * sc, a = st.a * sc, sr = st.sr * scr, b = st.b * scr;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (FULL || j < nv) {
                // two rounded products, so that identical heads give d = 0 exactly; the
                // exponents reuse them (x k - m k)
                const float xk = __fmul_rn(x[j], k), xrk = __fmul_rn(xr[j], kr);
                const float d = xk - xrk;
                const float e = ex2_approx(xk - nmk);
                const float er = ex2_approx(xrk - nmrk);
                s += e;
                a = fmaf(e, d, a);
                sr += er;
                b = fmaf(er, -d, b);
            }
        }
        st.m = nm;
        st.s = s;
        st.a = a;
        st.mr = nmr;
        st.sr = sr;
        st.b = b;
    }

    __device__ void epi_end(int u, int row, int half, EpiState& st) const {
        int m, c;
        unit(u, m, c);
        const int t = m * kTileM + row;
        if (t >= N) return;
        const size_t o = (static_cast<size_t>(c) * 2 + half) * N + t;
        part_p[o] = make_float2(st.m, st.s);
        part_a[o] = st.a;
        part_r[o] = make_float2(st.mr, st.sr);
        part_b[o] = st.b;
        if (st.found) s_target[t] = st.sy;
    }
};

__global__ void kl_merge_kernel(const float2* __restrict__ part_p, const float* __restrict__ part_a,
                                const float2* __restrict__ part_r, const float* __restrict__ part_b,
                                const float* __restrict__ s_target,
                                const int64_t* __restrict__ targets,
                                const uint8_t* __restrict__ mask, int N, int V, int num_parts,
                                float k, float kr, float* __restrict__ kl,
                                float* __restrict__ kl_rev, float* __restrict__ lse,
                                float* __restrict__ lse_ref, float* __restrict__ logp,
                                uint32_t* err) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= N) return;
    if (mask != nullptr && mask[t] == 0) {
        kl[t] = 0.f;
        if (kl_rev != nullptr) kl_rev[t] = 0.f;
        if (lse != nullptr) lse[t] = 0.f;
        if (lse_ref != nullptr) lse_ref[t] = 0.f;
        if (logp != nullptr) logp[t] = 0.f;
        return;
    }
    // parts in ascending (chunk, column half) order
    float m = -INFINITY, mr = -INFINITY;
    for (int c = 0; c < num_parts; ++c) {
        m = fmaxf(m, part_p[static_cast<size_t>(c) * N + t].x);
        mr = fmaxf(mr, part_r[static_cast<size_t>(c) * N + t].x);
    }
    float s = 0.f, a = 0.f, sr = 0.f, b = 0.f;
    for (int c = 0; c < num_parts; ++c) {
        const size_t o = static_cast<size_t>(c) * N + t;
        const float2 pp = part_p[o], pr = part_r[o];
        const float w = ex2_approx((pp.x - m) * k), wr = ex2_approx((pr.x - mr) * kr);
        s += pp.y * w;
        a += part_a[o] * w;
        sr += pr.y * wr;
        b += part_b[o] * wr;
    }
    const float lse2 = m * k + lg2_approx(s);
    const float lse2r = mr * kr + lg2_approx(sr);
    // the same expression for both directions, so that swapping the heads swaps them bitwise
    kl[t] = (a / s + (lse2r - lse2)) * kLn2f;
    if (kl_rev != nullptr) kl_rev[t] = (b / sr + (lse2 - lse2r)) * kLn2f;
    if (lse != nullptr) lse[t] = lse2 * kLn2f;
    if (lse_ref != nullptr) lse_ref[t] = lse2r * kLn2f;
    if (logp != nullptr) {
        const int64_t y = targets[t];
        if (y < 0 || y >= V) {
            logp[t] = __int_as_float(0x7fc00000);
            if (err != nullptr) atomicOr(err, RLK_DEVERR_TARGET_RANGE);
        } else {
            logp[t] = (s_target[t] * k - lse2) * kLn2f;
        }
    }
}

}  // namespace

cudaError_t launch_kl_fwd(const CUtensorMap& map_h, const CUtensorMap& map_w,
                          const CUtensorMap& map_hr, const CUtensorMap& map_wr,
                          const int64_t* targets, const uint8_t* mask, int N, int H, int Hr, int V,
                          float k, float kr, float* kl, float* kl_rev, float* lse, float* lse_ref,
                          float* logp, void* workspace, uint32_t* err, int num_sms,
                          cudaStream_t stream) {
    const KlFwdLayout lay(N, V);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    KlFwdPolicy p;
    p.targets = logp != nullptr ? targets : nullptr;
    p.part_p = reinterpret_cast<float2*>(ws + lay.part_p_off);
    p.part_a = reinterpret_cast<float*>(ws + lay.part_a_off);
    p.part_r = reinterpret_cast<float2*>(ws + lay.part_r_off);
    p.part_b = reinterpret_cast<float*>(ws + lay.part_b_off);
    p.s_target = reinterpret_cast<float*>(ws + lay.target_off);
    p.N = N;
    p.V = V;
    p.num_m = (N + kTileM - 1) / kTileM;
    p.num_vt = (V + kTileV - 1) / kTileV;
    p.num_chunks = static_cast<int>(lay.num_chunks);
    p.kblocks = H / 64;
    p.kblocks_r = Hr / 64;
    p.k = k;
    p.kr = kr;
    auto kern = gemm_persistent_kernel<KlFwdPolicy>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kGemmSmemBytes));
    if (e != cudaSuccess) return e;
    const long long units = static_cast<long long>(p.num_m) * p.num_chunks;
    const int grid = static_cast<int>(units < num_sms ? units : num_sms);
    kern<<<grid, gemm_threads<KlFwdPolicy>(), kGemmSmemBytes, stream>>>(
        KlMaps{map_h, map_w, map_hr, map_wr}, p, err, 0u);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    kl_merge_kernel<<<(N + 255) / 256, 256, 0, stream>>>(
        p.part_p, p.part_a, p.part_r, p.part_b, p.s_target, targets, mask, N, V,
        2 * p.num_chunks, k, kr, kl, kl_rev, lse, lse_ref, logp, err);
    return cudaGetLastError();
}

}  // namespace rlk
