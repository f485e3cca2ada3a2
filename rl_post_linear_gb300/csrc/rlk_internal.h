// rlk_internal.h -- constants and launcher declarations shared by the
// translation units of the CUDA library (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/rlk.h"

namespace rlk {

// Fixed numeric contract.  None of these may depend on N, the mask or the GPU.
constexpr int kTileM = 128;                 // tokens per accumulator tile
constexpr int kTileV = 256;                 // vocab (or hidden) columns per tile
constexpr int kFwdTilesPerChunk = 4;        // forward vocab chunk = 1024 columns
constexpr int kFwdChunk = kFwdTilesPerChunk * kTileV;
constexpr int kBwdChunk = 32768;            // backward vocab chunk (multiple of kTileV)
constexpr int kMaxBwdChunks = 65536;        // 2^31 / kBwdChunk: chunks of the largest vocabulary
// Raster groups (visiting order only; no effect on any result): token rows per
// group for the forward and dS GEMMs, hidden tiles per group for the dW GEMM.
// A group's share of h (4096 rows, or 8 x 256 columns, of H = 4096) is 33.5 MB,
// which stays resident in L2 while the other operand streams.
constexpr int kRasterTokenRows = 4096;
constexpr int kRasterHiddenTiles = 8;
// Rows of the tile a CTA pair computes (the forward, dS, dh and dW GEMMs).  Each
// CTA of the pair loads half of the tile's B operand: K-major B tensor maps of
// these GEMMs have boxes of kPairBRows rows (their ring slots hold no more).
constexpr int kUnitM = 256;
constexpr int kPairBRows = kTileV / 2;
constexpr int kAuditThreads = 256;
constexpr int kLossPerThread = 16;          // 4 float4 of each input per thread (loss fragment)
constexpr int kAuditV3PerThread = 16;       // 4 float4 of each input per thread (audit)
constexpr int kLossBlockElems = kAuditThreads * kLossPerThread;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Forward workspace: per (vocab chunk, row) partials {max s, sum 2^((s-max)k)},
// then the target logit per row.
// (With entropy, a third per (chunk, row) partial: sum 2^((s-max)k) s.)  For a
// masked batch the active rows are compacted first: the row lists, the active
// count and the compacted copy of h [N, H] follow.
constexpr int kCompactBlock = 1024;
struct FwdLayout {
    int64_t num_chunks;
    size_t partial_off, partial_a_off, target_off, rows_off, pos_off, blk_off, count_off, hc_off,
        total;
    FwdLayout(int64_t N, int64_t H, int64_t V) {
        const int64_t vt = (V + kTileV - 1) / kTileV;
        num_chunks = (vt + kFwdTilesPerChunk - 1) / kFwdTilesPerChunk;
        partial_off = 0;
        partial_a_off = align_up(static_cast<size_t>(num_chunks) * N * 8, 256);
        target_off = align_up(partial_a_off + static_cast<size_t>(num_chunks) * N * 4, 256);
        rows_off = align_up(target_off + static_cast<size_t>(N) * 4, 256);
        pos_off = align_up(rows_off + static_cast<size_t>(N) * 4, 256);
        blk_off = align_up(pos_off + static_cast<size_t>(N) * 4, 256);
        count_off = align_up(blk_off + static_cast<size_t>((N + kCompactBlock - 1) / kCompactBlock) * 4, 256);
        hc_off = align_up(count_off + 4, 256);
        total = align_up(hc_off + static_cast<size_t>(N) * H * 2, 256);
    }
};

// Backward workspace: dS for one vocab chunk [N, kBwdChunk] bf16 (hilo: a hi
// and a lo plane, [N, 2 kBwdChunk]), the fp32 dh accumulator [N, H], the
// (target, token) list sorted by target, 1 - p_y per row, each row's dominant
// non-target class and the chunk's (class, token) list sorted by class, and the
// sorted key tiles the lists are built from.
constexpr int kTargetSortTile = 2048;
struct BwdLayout {
    size_t ds_off, dhacc_off, sorted_y_off, sorted_t_off, ycoef_off, dom_off, dcoef_off,
        sorted_dy_off, sorted_dt_off, tiles_off, blk_off, rows_off, pos_off, count_off, hc_off,
        flags_off, total;
    BwdLayout(int64_t N, int64_t H, bool hilo = false) {
        ds_off = 0;
        dhacc_off = align_up(static_cast<size_t>(N) * kBwdChunk * 2 * (hilo ? 2 : 1), 256);
        sorted_y_off = align_up(dhacc_off + static_cast<size_t>(N) * H * 4, 256);
        sorted_t_off = align_up(sorted_y_off + static_cast<size_t>(N) * 4, 256);
        ycoef_off = align_up(sorted_t_off + static_cast<size_t>(N) * 4, 256);
        dom_off = align_up(ycoef_off + static_cast<size_t>(N) * 4, 256);
        dcoef_off = align_up(dom_off + static_cast<size_t>(N) * 4, 256);
        sorted_dy_off = align_up(dcoef_off + static_cast<size_t>(N) * 4, 256);
        sorted_dt_off = align_up(sorted_dy_off + static_cast<size_t>(N) * 4, 256);
        tiles_off = align_up(sorted_dt_off + static_cast<size_t>(N) * 4, 256);
        const size_t tiles = static_cast<size_t>((N + kTargetSortTile - 1) / kTargetSortTile);
        // compaction of a masked batch, as in the forward
        blk_off = align_up(tiles_off + tiles * kTargetSortTile * 8, 256);
        rows_off = align_up(blk_off + static_cast<size_t>((N + kCompactBlock - 1) / kCompactBlock) * 4,
                            256);
        pos_off = align_up(rows_off + static_cast<size_t>(N) * 4, 256);
        count_off = align_up(pos_off + static_cast<size_t>(N) * 4, 256);
        hc_off = align_up(count_off + 4, 256);
        // one flag per vocab chunk: the chunk holds some token's dominant class
        flags_off = align_up(hc_off + static_cast<size_t>(N) * H * 2, 256);
        total = align_up(flags_off + static_cast<size_t>(kMaxBwdChunks) * 4, 256);
    }
};

// A sum carried as an unevaluated pair of floats (hi + lo, about 48 significant
// bits), added with Knuth's two-sum: the audit's cross-block accumulation.  The
// fp64 units of this GPU are few and slow; pairs of fp32 operations are not.
struct DFloat {
    float hi, lo;
};

struct AuditPartial {
    int64_t count;
    int64_t arg;
    DFloat sum_d;
    DFloat sum_kl;
    float best;
    uint32_t flags;
};

struct LossPartial {
    int64_t count;
    int64_t clipped;
    int64_t outside;
    double sum_term;
    double sum_r;
};

inline size_t loss_blocks(int64_t N) {
    return static_cast<size_t>((N + kLossBlockElems - 1) / kLossBlockElems);
}

inline size_t audit_v3_blocks(int64_t N) {
    const int64_t b = kAuditThreads * kAuditV3PerThread;
    return static_cast<size_t>((N + b - 1) / b);
}

// Launchers (return the first CUDA error, cudaSuccess otherwise).
// Full-vocabulary KL forward workspace: per (1024-column chunk, column half of
// its tiles, row) the policy's (max, sum) float2 and sum of weighted
// log-ratios, the same for the reference, and the policy's target logit per row.
struct KlFwdLayout {
    int64_t num_chunks;
    size_t part_p_off, part_a_off, part_r_off, part_b_off, target_off, total;
    KlFwdLayout(int64_t N, int64_t V) {
        const int64_t vt = (V + kTileV - 1) / kTileV;
        num_chunks = (vt + kFwdTilesPerChunk - 1) / kFwdTilesPerChunk;
        const size_t cn = static_cast<size_t>(num_chunks) * 2 * N;
        part_p_off = 0;
        part_a_off = align_up(cn * 8, 256);
        part_r_off = align_up(part_a_off + cn * 4, 256);
        part_b_off = align_up(part_r_off + cn * 8, 256);
        target_off = align_up(part_b_off + cn * 4, 256);
        total = align_up(target_off + static_cast<size_t>(N) * 4, 256);
    }
};

cudaError_t launch_kl_fwd(const CUtensorMap& map_h, const CUtensorMap& map_w,
                          const CUtensorMap& map_hr, const CUtensorMap& map_wr,
                          const int64_t* targets, const uint8_t* mask, int N, int H, int Hr, int V,
                          float k, float kr, float* kl, float* kl_rev, float* lse, float* lse_ref,
                          float* logp, void* workspace, uint32_t* err, int num_sms,
                          cudaStream_t stream);

// rows / n_rows / pos_of: the compaction of a masked batch (all nullptr when the
// GEMM runs over the original rows).
cudaError_t launch_fwd(const CUtensorMap& map_h, const CUtensorMap& map_w,
                       const int64_t* targets, const uint8_t* mask, int N, int H, int V,
                       float k_log2e_over_t, float* logp, float* lse, float* entropy,
                       void* workspace, const int* rows, const int* n_rows, const int* pos_of,
                       uint32_t* err, int num_sms, cudaStream_t stream);

cudaError_t launch_compact(const uint8_t* mask, int N, int H, const void* hidden, void* hidden_c,
                           int* blk_count, int* rows, int* pos_of, int* n_active,
                           cudaStream_t stream);
// zeroes the rows (row_bytes each, a multiple of 16) of the tokens with mask 0
cudaError_t launch_zero_inactive_rows(const uint8_t* mask, int N, size_t row_bytes, void* out,
                                      cudaStream_t stream);

cudaError_t launch_fwd_partials(const CUtensorMap& map_h, const CUtensorMap& map_w,
                                const int64_t* targets, const uint8_t* mask, int N, int H,
                                int V_local, int64_t vocab_start, float k, float2* partials,
                                float* s_target, uint32_t* err, int num_sms, cudaStream_t stream);

cudaError_t launch_fwd_merge(const float2* partials, int num_chunks, const float* s_target,
                             const int64_t* targets, const uint8_t* mask, int N, int V, float k,
                             float* logp, float* lse, uint32_t* err, cudaStream_t stream);

inline int64_t fwd_num_chunks(int64_t V) {
    return ((V + kTileV - 1) / kTileV + kFwdTilesPerChunk - 1) / kFwdTilesPerChunk;
}

// Tensor maps of the backward launches (one role per launch).
struct BwdStepMaps {
    CUtensorMap h_kmajor;      // hidden [N,H], box {64, 128}: A of the dS recompute
    CUtensorMap w_kmajor;      // weight [V,H], box {64, 128}: B of the KL dS recompute (pair)
    CUtensorMap w_kmajor_pair; // weight [V,H], box {64, 128}: B of the dS recompute (CTA pair)
    CUtensorMap w_mnmajor;     // weight [V,H], box {64, 64}:  B of the dh GEMM
    CUtensorMap h_mnmajor;     // hidden [N,H], box {64, 64}:  B of the dW GEMM
    CUtensorMap ds_kmajor;     // consumed dS [N, width], box {64, 128}: A of the dh GEMM
    CUtensorMap ds_mnmajor;    // consumed dS [N, width], box {64, 64}:  A of the dW GEMM
    CUtensorMap hr_kmajor;     // KL only: reference hidden [N,Hr], box {64, 128}
    CUtensorMap wr_kmajor;     // KL only: reference weight [V,Hr], box {64, 128} (pair)
    CUtensorMap ds_store;      // KL only: dS [N, width] written by TMA stores, box {32, 32}
};

// One launch of the backward: a role (the dS recompute, the dh GEMM or the dW
// GEMM) over one vocabulary chunk.
constexpr int kRoleDs = 0, kRoleDh = 1, kRoleDw = 2;
struct BwdStep {
    const int64_t* targets;
    const uint8_t* mask;
    const float* grad;
    const float* grad_ent;     // entropy gradient, or nullptr
    const float* ent;          // forward entropy, or nullptr
    const float* lse;
    const void* hidden;
    const void* weight;
    int N, H, V, num_chunks;       // V: rows of the weight (block) being differentiated
    int chunk, role;
    float k, temp;
    int64_t y_off;             // global id of the weight block's first row (0 unsharded)
    int V_global;              // vocabulary size
    bool round_last;           // false: the fp32 partial of dh goes to dh_out32, unrounded
    float* dh_out32;           // [N][H] by token (round_last false)
    float* dw_out32;           // non-null: dW as an unrounded fp32 partial [V][H]
    const int* rows;           // compaction of a masked batch: row -> token, or nullptr
    const int* n_rows;         // number of compacted rows (device), or nullptr
    // KL against a reference head (kl = true): dS from both heads, no fp32 target terms
    bool kl;
    int H_ref;
    float k_ref;
    const float* grad_rev;     // d loss / d KL(q || p), or nullptr
    const float* lse_ref;
    const float* kl_val;       // the forward's KL(p || q)
    bool hilo;                 // dS as hi and lo bf16 planes [N, 2 kBwdChunk] (entropy, KL)
    void* ds;                  // dS [N, kBwdChunk] bf16 of the chunk (hilo: [N, 2 kBwdChunk])
    float* dh_acc;
    const int* sorted_y;
    const int* sorted_t;
    float* ycoef;              // [N] 1 - p_y of each live row
    int* dom;                  // [N] dominant non-target class (p > 1/2) or -1
    int* dom_flags;            // [num_chunks] nonzero: the chunk holds some row's dominant class
    float* dcoef;              // [N] its fp32 gradient coefficient
    int* sorted_dy;            // [N] this chunk's dominant classes, ascending (V: none)
    int* sorted_dt;            // [N]
    uint64_t* tiles;           // sort scratch
    void* dhidden;
    void* dweight;
};

cudaError_t launch_target_sort(const int64_t* targets, const uint8_t* mask, int N, int V,
                               int64_t y_off, int V_global, uint64_t* tiles, int* sorted_y,
                               int* sorted_t, int* dom, int* dom_flags, int num_chunks, uint32_t* err,
                               cudaStream_t stream);

cudaError_t launch_dh_merge(const float* partials, int64_t num_parts, int64_t N, int64_t H,
                            void* dhidden, cudaStream_t stream);

cudaError_t launch_bwd_step(const BwdStepMaps& maps, const BwdStep& step, int num_sms,
                            uint32_t* err, cudaStream_t stream);

// The audit: per-block partials (at most 608 of them), then their merge in a fixed
// order by a second launch.  vec_ok: new / old 16-byte and the mask 4-byte aligned
// (vector loads).
cudaError_t launch_audit(const float* logp_new, const float* logp_old, const uint8_t* mask,
                         int64_t N, rlk_audit_result_t* result, void* partials, bool vec_ok,
                         cudaStream_t stream);

cudaError_t launch_grpo_loss(const float* logp_new, const float* logp_old, const float* adv,
                             const uint8_t* mask, int64_t N, double eps_low, double eps_high,
                             double scale, float* grad, rlk_grpo_result_t* result,
                             void* workspace, bool vec_ok, cudaStream_t stream);

cudaError_t launch_logp_from_logits(const void* logits, bool bf16, int64_t stride, int64_t N, int V,
                                    const int64_t* rows, int M, const int64_t* targets,
                                    const uint8_t* mask, float k, bool vec_ok, float* logp,
                                    float* lse, uint32_t* err, cudaStream_t stream);

size_t audit_ext_workspace(int64_t N);
cudaError_t launch_audit_ext(const float* logp_new, const float* logp_old, const uint8_t* mask,
                             int64_t N, const int64_t* seq_offsets, int64_t num_seqs, float eps,
                             rlk_audit_ext_t* result, void* workspace, bool vec_ok, int sms,
                             cudaStream_t stream);

// Device address (current device and context) of the library-owned audit scratch.
cudaError_t audit_noalloc_scratch(void** parts);

}  // namespace rlk
