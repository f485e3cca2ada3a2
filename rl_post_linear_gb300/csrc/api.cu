// api.cu -- the C ABI (include/rlk.h): argument validation, TMA tensor maps,
// and the launch sequence of each entry point.  Every argument error is
// detected on the host before anything is enqueued, so invalid calls never
// reach the GPU.  The library allocates nothing and never synchronises.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <mutex>

#include "rlk_internal.h"

namespace {

using rlk::align_up;

// 32-bit device indices, with headroom for rounding N and V up to whole tiles
constexpr int64_t kMaxDim = (int64_t(1) << 31) - (int64_t(1) << 16);

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

struct DeviceInfo {
    int sms = 0;
    bool supported = false;
    bool valid = false;
};

// SM count and architecture of the current device (queried once per device).
rlk_status_t current_device(DeviceInfo& out) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return RLK_ERR_LAUNCH;
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo& d = cache[dev];
    if (!d.valid) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return RLK_ERR_LAUNCH;
        d.sms = sms;
        d.supported = (major == 10 && minor == 3);
        d.valid = true;
    }
    out = d;
    return out.supported ? RLK_OK : RLK_ERR_UNSUPPORTED;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// 2D bf16 tensor map, 128-byte swizzle, zero fill outside the tensor.
rlk_status_t make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                      uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                      CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return RLK_ERR_LAUNCH;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? RLK_OK : RLK_ERR_LAUNCH;
}

rlk_status_t check_shape(int64_t N, int64_t H, int64_t V, double temperature) {
    if (N < 0 || N > kMaxDim || V < 1 || V > kMaxDim || H < 1) return RLK_ERR_INVALID_VALUE;
    if (!(std::isfinite(temperature) && temperature > 0.0)) return RLK_ERR_INVALID_VALUE;
    if (H % 64 != 0 || H > (int64_t(1) << 24)) return RLK_ERR_UNSUPPORTED;
    return RLK_OK;
}

#define RLK_TRY(expr)                        \
    do {                                     \
        rlk_status_t s_ = (expr);            \
        if (s_ != RLK_OK) return s_;         \
    } while (0)

#define RLK_CUDA(expr)                                    \
    do {                                                  \
        if ((expr) != cudaSuccess) return RLK_ERR_LAUNCH; \
    } while (0)

}  // namespace

extern "C" {

size_t rlk_linear_logp_fwd_workspace_bytes(int64_t N, int64_t H, int64_t V) {
    if (N < 0 || V < 1 || H < 0) return 0;
    return rlk::FwdLayout(N, H, V).total;
}

size_t rlk_linear_logp_bwd_workspace_bytes(int64_t N, int64_t H, int64_t V) {
    (void)V;
    if (N < 0 || H < 0) return 0;
    return rlk::BwdLayout(N, H).total;
}

size_t rlk_linear_logp_entropy_bwd_workspace_bytes(int64_t N, int64_t H, int64_t V) {
    (void)V;
    if (N < 0 || H < 0) return 0;
    return rlk::BwdLayout(N, H, true).total;
}

size_t rlk_dlogp_audit_workspace_bytes(int64_t N) {
    if (N < 0) return 0;
    return align_up(rlk::audit_v3_blocks(N) * sizeof(rlk::AuditPartial), 256) + 256;
}

// The vocabulary in ascending kBwdChunk-column chunks; per chunk the dS
// recompute, then the dh and the dW GEMMs, one launch per role (the roles of a
// chunk share L2 best when each has the GPU to itself).
static rlk_status_t bwd_chunks(rlk::BwdStepMaps& maps, rlk::BwdStep& st, void* ds, int64_t N,
                               int64_t V, int sms, uint32_t* device_error_word,
                               cudaStream_t stream) {
    // hilo: each dS row holds the hi plane, then the lo plane kBwdChunk columns on; the
    // maps span both (the columns between them are written or never read)
    const uint64_t ld = uint64_t(rlk::kBwdChunk) * (st.hilo ? 2 : 1);
    for (int c = 0; c < st.num_chunks; ++c) {
        const int64_t width = std::min<int64_t>(rlk::kBwdChunk, V - int64_t(c) * rlk::kBwdChunk);
        const uint64_t inner = uint64_t(width) + (st.hilo ? uint64_t(rlk::kBwdChunk) : 0);
        RLK_TRY(make_map(&maps.ds_kmajor, ds, inner, N, ld * 2, 64, rlk::kTileM));
        RLK_TRY(make_map(&maps.ds_mnmajor, ds, inner, N, ld * 2, 64, 64));
        if (st.kl)   // the KL dS epilogue writes its tiles with TMA stores
            RLK_TRY(make_map(&maps.ds_store, ds, inner, N, ld * 2, 32, 32,
                             CU_TENSOR_MAP_SWIZZLE_NONE));
        st.ds = ds;
        st.chunk = c;
        for (int role : {rlk::kRoleDs, rlk::kRoleDh, rlk::kRoleDw}) {
            st.role = role;
            RLK_CUDA(rlk::launch_bwd_step(maps, st, sms, device_error_word, stream));
        }
    }
    return RLK_OK;
}

static rlk_status_t fwd_impl(const void* hidden, const void* weight, const int64_t* targets,
                             const uint8_t* active_mask, int64_t N, int64_t H, int64_t V,
                             double temperature, float* logp_out, float* lse_out,
                             float* entropy_out, void* workspace, size_t workspace_bytes,
                             uint32_t* device_error_word, cudaStream_t stream) {
    RLK_TRY(check_shape(N, H, V, temperature));
    if (N == 0) return RLK_OK;
    if (hidden == nullptr || weight == nullptr || targets == nullptr || logp_out == nullptr)
        return RLK_ERR_INVALID_VALUE;
    if (!aligned(hidden, 16) || !aligned(weight, 16)) return RLK_ERR_INVALID_VALUE;
    if (workspace == nullptr || !aligned(workspace, 256) ||
        workspace_bytes < rlk_linear_logp_fwd_workspace_bytes(N, H, V))
        return RLK_ERR_WORKSPACE;
    DeviceInfo dev;
    RLK_TRY(current_device(dev));

    // a masked batch is compacted to its active rows first (ascending token order)
    const rlk::FwdLayout lay(N, H, V);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* rows = nullptr;
    int* pos_of = nullptr;
    int* n_rows = nullptr;
    const void* gemm_rows = hidden;
    if (active_mask != nullptr) {
        rows = reinterpret_cast<int*>(ws + lay.rows_off);
        pos_of = reinterpret_cast<int*>(ws + lay.pos_off);
        n_rows = reinterpret_cast<int*>(ws + lay.count_off);
        void* hc = ws + lay.hc_off;
        RLK_CUDA(rlk::launch_compact(active_mask, static_cast<int>(N), static_cast<int>(H), hidden,
                                     hc, reinterpret_cast<int*>(ws + lay.blk_off), rows, pos_of,
                                     n_rows, stream));
        gemm_rows = hc;
    }
    CUtensorMap map_h, map_w;
    RLK_TRY(make_map(&map_h, gemm_rows, H, N, H * 2, 64, rlk::kTileM));
    RLK_TRY(make_map(&map_w, weight, H, V, H * 2, 64, rlk::kPairBRows));
    const float k = static_cast<float>(1.4426950408889634074 / temperature);
    RLK_CUDA(rlk::launch_fwd(map_h, map_w, targets, active_mask, static_cast<int>(N),
                             static_cast<int>(H), static_cast<int>(V), k, logp_out, lse_out,
                             entropy_out, workspace, rows, n_rows, pos_of, device_error_word,
                             dev.sms, stream));
    return RLK_OK;
}

rlk_status_t rlk_linear_logp_fwd(const void* hidden, const void* weight, const int64_t* targets,
                                 const uint8_t* active_mask, int64_t N, int64_t H, int64_t V,
                                 double temperature, float* logp_out, float* lse_out,
                                 void* workspace, size_t workspace_bytes,
                                 uint32_t* device_error_word, cudaStream_t stream) {
    return fwd_impl(hidden, weight, targets, active_mask, N, H, V, temperature, logp_out, lse_out,
                    nullptr, workspace, workspace_bytes, device_error_word, stream);
}

size_t rlk_linear_kl_fwd_workspace_bytes(int64_t N, int64_t V) {
    if (N < 0 || V < 1) return 0;
    return rlk::KlFwdLayout(N, V).total;
}

rlk_status_t rlk_linear_kl_fwd(const void* hidden, const void* weight, const void* hidden_ref,
                               const void* weight_ref, const int64_t* targets,
                               const uint8_t* active_mask, int64_t N, int64_t H, int64_t H_ref,
                               int64_t V, double temperature, double temperature_ref,
                               float* kl_out, float* kl_rev_out, float* lse_out,
                               float* lse_ref_out, float* logp_out, void* workspace,
                               size_t workspace_bytes, uint32_t* device_error_word,
                               cudaStream_t stream) {
    RLK_TRY(check_shape(N, H, V, temperature));
    RLK_TRY(check_shape(N, H_ref, V, temperature_ref));
    if (N == 0) return RLK_OK;
    if (hidden == nullptr || weight == nullptr || hidden_ref == nullptr ||
        weight_ref == nullptr || kl_out == nullptr)
        return RLK_ERR_INVALID_VALUE;
    if (logp_out != nullptr && targets == nullptr) return RLK_ERR_INVALID_VALUE;
    if (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(hidden_ref, 16) ||
        !aligned(weight_ref, 16))
        return RLK_ERR_INVALID_VALUE;
    if (workspace == nullptr || !aligned(workspace, 256) ||
        workspace_bytes < rlk_linear_kl_fwd_workspace_bytes(N, V))
        return RLK_ERR_WORKSPACE;
    DeviceInfo dev;
    RLK_TRY(current_device(dev));
    CUtensorMap map_h, map_w, map_hr, map_wr;
    RLK_TRY(make_map(&map_h, hidden, H, N, H * 2, 64, rlk::kTileM));
    RLK_TRY(make_map(&map_w, weight, H, V, H * 2, 64, rlk::kTileV));
    RLK_TRY(make_map(&map_hr, hidden_ref, H_ref, N, H_ref * 2, 64, rlk::kTileM));
    RLK_TRY(make_map(&map_wr, weight_ref, H_ref, V, H_ref * 2, 64, rlk::kTileV));
    const float k = static_cast<float>(1.4426950408889634074 / temperature);
    const float kr = static_cast<float>(1.4426950408889634074 / temperature_ref);
    RLK_CUDA(rlk::launch_kl_fwd(map_h, map_w, map_hr, map_wr, targets, active_mask,
                                static_cast<int>(N), static_cast<int>(H),
                                static_cast<int>(H_ref), static_cast<int>(V), k, kr, kl_out,
                                kl_rev_out, lse_out, lse_ref_out, logp_out, workspace,
                                device_error_word, dev.sms, stream));
    return RLK_OK;
}

size_t rlk_linear_kl_bwd_workspace_bytes(int64_t N, int64_t H, int64_t V) {
    return rlk_linear_logp_entropy_bwd_workspace_bytes(N, H, V);
}

rlk_status_t rlk_linear_kl_bwd(const void* hidden, const void* weight, const void* hidden_ref,
                               const void* weight_ref, const uint8_t* active_mask,
                               const float* grad_kl, const float* grad_kl_rev, const float* lse,
                               const float* lse_ref, const float* kl, int64_t N, int64_t H,
                               int64_t H_ref, int64_t V, double temperature,
                               double temperature_ref, void* dhidden, void* dweight,
                               void* workspace, size_t workspace_bytes,
                               uint32_t* device_error_word, cudaStream_t stream) {
    RLK_TRY(check_shape(N, H, V, temperature));
    RLK_TRY(check_shape(N, H_ref, V, temperature_ref));
    if (N == 0) return RLK_OK;
    if (hidden == nullptr || weight == nullptr || hidden_ref == nullptr ||
        weight_ref == nullptr || lse == nullptr || lse_ref == nullptr || dhidden == nullptr ||
        dweight == nullptr || (grad_kl == nullptr && grad_kl_rev == nullptr) ||
        (grad_kl != nullptr && kl == nullptr))
        return RLK_ERR_INVALID_VALUE;
    if (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(hidden_ref, 16) ||
        !aligned(weight_ref, 16) || !aligned(dhidden, 16) || !aligned(dweight, 16))
        return RLK_ERR_INVALID_VALUE;
    if (workspace == nullptr || !aligned(workspace, 256) ||
        workspace_bytes < rlk_linear_kl_bwd_workspace_bytes(N, H, V))
        return RLK_ERR_WORKSPACE;
    DeviceInfo dev;
    RLK_TRY(current_device(dev));

    const rlk::BwdLayout lay(N, H, true);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    rlk::BwdStepMaps maps;
    RLK_TRY(make_map(&maps.h_kmajor, hidden, H, N, H * 2, 64, rlk::kTileM));
    RLK_TRY(make_map(&maps.w_kmajor, weight, H, V, H * 2, 64, rlk::kPairBRows));
    RLK_TRY(make_map(&maps.w_mnmajor, weight, H, V, H * 2, 64, 64));
    RLK_TRY(make_map(&maps.h_mnmajor, hidden, H, N, H * 2, 64, 64));
    RLK_TRY(make_map(&maps.hr_kmajor, hidden_ref, H_ref, N, H_ref * 2, 64, rlk::kTileM));
    RLK_TRY(make_map(&maps.wr_kmajor, weight_ref, H_ref, V, H_ref * 2, 64, rlk::kPairBRows));
    rlk::BwdStep st{};
    st.mask = active_mask;
    st.grad = grad_kl;
    st.lse = lse;
    st.hidden = hidden;
    st.weight = weight;
    st.N = static_cast<int>(N);
    st.H = static_cast<int>(H);
    st.V = static_cast<int>(V);
    st.num_chunks = static_cast<int>((V + rlk::kBwdChunk - 1) / rlk::kBwdChunk);
    st.k = static_cast<float>(1.4426950408889634074 / temperature);
    st.temp = static_cast<float>(temperature);
    st.kl = true;
    st.hilo = true;
    st.y_off = 0;
    st.V_global = static_cast<int>(V);
    st.round_last = true;
    st.H_ref = static_cast<int>(H_ref);
    st.k_ref = static_cast<float>(1.4426950408889634074 / temperature_ref);
    st.grad_rev = grad_kl_rev;
    st.lse_ref = lse_ref;
    st.kl_val = kl;
    st.dh_acc = reinterpret_cast<float*>(ws + lay.dhacc_off);
    st.dom = reinterpret_cast<int*>(ws + lay.dom_off);
    st.dom_flags = reinterpret_cast<int*>(ws + lay.flags_off);
    st.dcoef = reinterpret_cast<float*>(ws + lay.dcoef_off);
    st.sorted_dy = reinterpret_cast<int*>(ws + lay.sorted_dy_off);
    st.sorted_dt = reinterpret_cast<int*>(ws + lay.sorted_dt_off);
    st.tiles = reinterpret_cast<uint64_t*>(ws + lay.tiles_off);
    st.dhidden = dhidden;
    st.dweight = dweight;
    // no dominant class yet (all bits set: -1), and none in any chunk
    RLK_CUDA(cudaMemsetAsync(st.dom, 0xff, static_cast<size_t>(N) * sizeof(int), stream));
    RLK_CUDA(cudaMemsetAsync(st.dom_flags, 0, static_cast<size_t>(st.num_chunks) * sizeof(int),
                             stream));
    return bwd_chunks(maps, st, ws + lay.ds_off, N, V, dev.sms, device_error_word, stream);
}

rlk_status_t rlk_linear_logp_entropy_fwd(const void* hidden, const void* weight,
                                         const int64_t* targets, const uint8_t* active_mask,
                                         int64_t N, int64_t H, int64_t V, double temperature,
                                         float* logp_out, float* lse_out, float* entropy_out,
                                         void* workspace, size_t workspace_bytes,
                                         uint32_t* device_error_word, cudaStream_t stream) {
    if (N > 0 && entropy_out == nullptr) return RLK_ERR_INVALID_VALUE;
    return fwd_impl(hidden, weight, targets, active_mask, N, H, V, temperature, logp_out, lse_out,
                    entropy_out, workspace, workspace_bytes, device_error_word, stream);
}

// The logp (and entropy) backward.  dh_partial == nullptr: the whole vocabulary,
// dh rounded to bf16 into dhidden.  Otherwise weight holds the rows
// [vocab_start, vocab_start + V) of a vocab_size-row head, and that block's fp32
// contribution to dh is written to dh_partial (dhidden unused).
static rlk_status_t bwd_impl(const void* hidden, const void* weight, const int64_t* targets,
                             const uint8_t* active_mask, const float* grad_logp,
                             const float* grad_entropy, const float* entropy, const float* lse,
                             int64_t N, int64_t H, int64_t V, int64_t vocab_start,
                             int64_t vocab_size, double temperature, void* dhidden,
                             float* dh_partial, void* dweight, float* dw_partial,
                             void* workspace, size_t workspace_bytes,
                             uint32_t* device_error_word, cudaStream_t stream) {
    RLK_TRY(check_shape(N, H, V, temperature));
    if (vocab_start < 0 || vocab_size > kMaxDim || vocab_start + V > vocab_size)
        return RLK_ERR_INVALID_VALUE;
    if (N == 0) return RLK_OK;
    void* dh_out = dh_partial != nullptr ? static_cast<void*>(dh_partial) : dhidden;
    void* dw_out = dw_partial != nullptr ? static_cast<void*>(dw_partial) : dweight;
    if (hidden == nullptr || weight == nullptr || targets == nullptr || grad_logp == nullptr ||
        lse == nullptr || dh_out == nullptr || dw_out == nullptr)
        return RLK_ERR_INVALID_VALUE;
    if (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(dh_out, 16) ||
        !aligned(dw_out, 16))
        return RLK_ERR_INVALID_VALUE;
    // the entropy gradient takes dS as hi / lo planes (twice the dS workspace)
    const bool hilo = grad_entropy != nullptr;
    const size_t need = hilo ? rlk_linear_logp_entropy_bwd_workspace_bytes(N, H, V)
                             : rlk_linear_logp_bwd_workspace_bytes(N, H, V);
    if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < need)
        return RLK_ERR_WORKSPACE;
    DeviceInfo dev;
    RLK_TRY(current_device(dev));

    const rlk::BwdLayout lay(N, H, hilo);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* dh_acc = reinterpret_cast<float*>(ws + lay.dhacc_off);
    int* sorted_y = reinterpret_cast<int*>(ws + lay.sorted_y_off);
    int* sorted_t = reinterpret_cast<int*>(ws + lay.sorted_t_off);
    const int n = static_cast<int>(N), h = static_cast<int>(H), v = static_cast<int>(V);

    // A masked batch runs its GEMMs over the active rows only (gathered in ascending
    // token order, as in the forward); the rows of dh of the inactive tokens are
    // zeroed here, since no GEMM visits them.
    int* rows = nullptr;
    int* n_rows = nullptr;
    const void* gemm_rows = hidden;
    if (active_mask != nullptr) {
        rows = reinterpret_cast<int*>(ws + lay.rows_off);
        n_rows = reinterpret_cast<int*>(ws + lay.count_off);
        void* hc = ws + lay.hc_off;
        RLK_CUDA(rlk::launch_compact(active_mask, n, h, hidden, hc,
                                     reinterpret_cast<int*>(ws + lay.blk_off), rows,
                                     reinterpret_cast<int*>(ws + lay.pos_off), n_rows, stream));
        RLK_CUDA(rlk::launch_zero_inactive_rows(
            active_mask, n, static_cast<size_t>(H) * (dh_partial != nullptr ? 4 : 2), dh_out,
            stream));
        gemm_rows = hc;
    }

    rlk::BwdStepMaps maps;
    RLK_TRY(make_map(&maps.h_kmajor, gemm_rows, H, N, H * 2, 64, rlk::kTileM));
    RLK_TRY(make_map(&maps.w_kmajor_pair, weight, H, V, H * 2, 64, rlk::kPairBRows));
    RLK_TRY(make_map(&maps.w_mnmajor, weight, H, V, H * 2, 64, 64));
    RLK_TRY(make_map(&maps.h_mnmajor, gemm_rows, H, N, H * 2, 64, 64));

    const int v_global = static_cast<int>(vocab_size);
    int* dom = reinterpret_cast<int*>(ws + lay.dom_off);
    uint64_t* tiles = reinterpret_cast<uint64_t*>(ws + lay.tiles_off);
    const int num_chunks = static_cast<int>((V + rlk::kBwdChunk - 1) / rlk::kBwdChunk);
    int* dom_flags = reinterpret_cast<int*>(ws + lay.flags_off);
    RLK_CUDA(rlk::launch_target_sort(targets, active_mask, n, v, vocab_start, v_global, tiles,
                                     sorted_y, sorted_t, dom, dom_flags, num_chunks,
                                     device_error_word, stream));
    rlk::BwdStep st{};
    st.targets = targets;
    st.mask = active_mask;
    st.grad = grad_logp;
    st.grad_ent = grad_entropy;
    st.ent = entropy;
    st.hilo = hilo;
    st.lse = lse;
    st.hidden = hidden;
    st.weight = weight;
    st.N = n;
    st.H = h;
    st.V = v;
    st.num_chunks = num_chunks;
    st.k = static_cast<float>(1.4426950408889634074 / temperature);
    st.temp = static_cast<float>(temperature);
    st.y_off = vocab_start;
    st.V_global = v_global;
    st.round_last = dh_partial == nullptr;
    st.dh_acc = dh_acc;
    st.dh_out32 = dh_partial;
    st.rows = rows;
    st.n_rows = n_rows;
    st.sorted_y = sorted_y;
    st.sorted_t = sorted_t;
    st.ycoef = reinterpret_cast<float*>(ws + lay.ycoef_off);
    st.dom = dom;
    st.dom_flags = dom_flags;
    st.dcoef = reinterpret_cast<float*>(ws + lay.dcoef_off);
    st.sorted_dy = reinterpret_cast<int*>(ws + lay.sorted_dy_off);
    st.sorted_dt = reinterpret_cast<int*>(ws + lay.sorted_dt_off);
    st.tiles = tiles;
    st.dhidden = dhidden;
    st.dweight = dweight;
    st.dw_out32 = dw_partial;
    return bwd_chunks(maps, st, ws + lay.ds_off, N, V, dev.sms, device_error_word, stream);
}

rlk_status_t rlk_linear_logp_bwd(const void* hidden, const void* weight, const int64_t* targets,
                                 const uint8_t* active_mask, const float* grad_logp,
                                 const float* lse, int64_t N, int64_t H, int64_t V,
                                 double temperature, void* dhidden, void* dweight,
                                 void* workspace, size_t workspace_bytes,
                                 uint32_t* device_error_word, cudaStream_t stream) {
    return bwd_impl(hidden, weight, targets, active_mask, grad_logp, nullptr, nullptr, lse, N, H,
                    V, 0, V, temperature, dhidden, nullptr, dweight, nullptr, workspace,
                    workspace_bytes, device_error_word, stream);
}

rlk_status_t rlk_linear_logp_bwd_dw_partial(const void* hidden, const void* weight,
                                            const int64_t* targets, const uint8_t* active_mask,
                                            const float* grad_logp, const float* lse, int64_t N,
                                            int64_t H, int64_t V, double temperature,
                                            void* dhidden, float* dweight_partial,
                                            void* workspace, size_t workspace_bytes,
                                            uint32_t* device_error_word, cudaStream_t stream) {
    if (N > 0 && dweight_partial == nullptr) return RLK_ERR_INVALID_VALUE;
    return bwd_impl(hidden, weight, targets, active_mask, grad_logp, nullptr, nullptr, lse, N, H,
                    V, 0, V, temperature, dhidden, nullptr, nullptr, dweight_partial, workspace,
                    workspace_bytes, device_error_word, stream);
}

rlk_status_t rlk_linear_logp_dw_merge(const float* dw_partials, int64_t num_partials, int64_t V,
                                      int64_t H, void* dweight, cudaStream_t stream) {
    if (num_partials < 1 || V < 0 || V > kMaxDim || H < 1) return RLK_ERR_INVALID_VALUE;
    if (H % 64 != 0) return RLK_ERR_UNSUPPORTED;
    if (V == 0) return RLK_OK;
    if (dw_partials == nullptr || dweight == nullptr || !aligned(dw_partials, 16) ||
        !aligned(dweight, 16))
        return RLK_ERR_INVALID_VALUE;
    RLK_CUDA(rlk::launch_dh_merge(dw_partials, num_partials, V, H, dweight, stream));
    return RLK_OK;
}

rlk_status_t rlk_linear_logp_bwd_shard(const void* hidden, const void* weight_shard,
                                       const int64_t* targets, const uint8_t* active_mask,
                                       const float* grad_logp, const float* lse, int64_t N,
                                       int64_t H, int64_t V_local, int64_t vocab_start,
                                       int64_t vocab_size, double temperature,
                                       float* dhidden_partial, void* dweight_shard,
                                       void* workspace, size_t workspace_bytes,
                                       uint32_t* device_error_word, cudaStream_t stream) {
    if (N > 0 && dhidden_partial == nullptr) return RLK_ERR_INVALID_VALUE;
    return bwd_impl(hidden, weight_shard, targets, active_mask, grad_logp, nullptr, nullptr, lse,
                    N, H, V_local, vocab_start, vocab_size, temperature, nullptr,
                    dhidden_partial, dweight_shard, nullptr, workspace, workspace_bytes,
                    device_error_word, stream);
}

rlk_status_t rlk_linear_logp_dh_merge(const float* dh_partials, int64_t num_partials, int64_t N,
                                      int64_t H, void* dhidden, cudaStream_t stream) {
    if (num_partials < 1 || N < 0 || N > kMaxDim || H < 1 || H % 64 != 0)
        return num_partials < 1 || N < 0 || N > kMaxDim || H < 1 ? RLK_ERR_INVALID_VALUE
                                                                 : RLK_ERR_UNSUPPORTED;
    if (N == 0) return RLK_OK;
    if (dh_partials == nullptr || dhidden == nullptr || !aligned(dh_partials, 16) ||
        !aligned(dhidden, 16))
        return RLK_ERR_INVALID_VALUE;
    RLK_CUDA(rlk::launch_dh_merge(dh_partials, num_partials, N, H, dhidden, stream));
    return RLK_OK;
}

rlk_status_t rlk_linear_logp_entropy_bwd(const void* hidden, const void* weight,
                                         const int64_t* targets, const uint8_t* active_mask,
                                         const float* grad_logp, const float* grad_entropy,
                                         const float* lse, const float* entropy, int64_t N,
                                         int64_t H, int64_t V, double temperature,
                                         void* dhidden, void* dweight, void* workspace,
                                         size_t workspace_bytes, uint32_t* device_error_word,
                                         cudaStream_t stream) {
    if (N > 0 && (grad_entropy == nullptr || entropy == nullptr)) return RLK_ERR_INVALID_VALUE;
    return bwd_impl(hidden, weight, targets, active_mask, grad_logp, grad_entropy, entropy, lse,
                    N, H, V, 0, V, temperature, dhidden, nullptr, dweight, nullptr, workspace,
                    workspace_bytes, device_error_word, stream);
}

rlk_status_t rlk_dlogp_audit(const float* logp_new, const float* logp_old,
                             const uint8_t* active_mask, int64_t N,
                             rlk_audit_result_t* result_dev, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
    if (N < 0 || N > (int64_t(1) << 40)) return RLK_ERR_INVALID_VALUE;
    if (result_dev == nullptr) return RLK_ERR_INVALID_VALUE;
    if (N > 0 && (logp_new == nullptr || logp_old == nullptr)) return RLK_ERR_INVALID_VALUE;
    if (workspace == nullptr || !aligned(workspace, 256) ||
        workspace_bytes < rlk_dlogp_audit_workspace_bytes(N))
        return RLK_ERR_WORKSPACE;
    DeviceInfo dev;
    RLK_TRY(current_device(dev));
    const bool vec_ok = aligned(logp_new, 16) && aligned(logp_old, 16) &&
                        (active_mask == nullptr || aligned(active_mask, 4));
    RLK_CUDA(rlk::launch_audit(logp_new, logp_old, active_mask, N, result_dev, workspace, vec_ok,
                               stream));
    return RLK_OK;
}

int64_t rlk_linear_logp_num_partials(int64_t V_local) {
    return V_local < 1 ? 0 : rlk::fwd_num_chunks(V_local);
}

rlk_status_t rlk_linear_logp_fwd_shard(const void* hidden, const void* weight_shard,
                                       const int64_t* targets, const uint8_t* active_mask,
                                       int64_t N, int64_t H, int64_t V_local,
                                       int64_t vocab_start, double temperature,
                                       float* partials_out, float* target_logit_out,
                                       uint32_t* device_error_word, cudaStream_t stream) {
    RLK_TRY(check_shape(N, H, V_local, temperature));
    if (vocab_start < 0 || vocab_start + V_local > kMaxDim) return RLK_ERR_INVALID_VALUE;
    if (vocab_start % rlk::kFwdChunk != 0) return RLK_ERR_UNSUPPORTED;
    if (N == 0) return RLK_OK;
    if (hidden == nullptr || weight_shard == nullptr || targets == nullptr ||
        partials_out == nullptr || target_logit_out == nullptr)
        return RLK_ERR_INVALID_VALUE;
    if (!aligned(hidden, 16) || !aligned(weight_shard, 16) || !aligned(partials_out, 8))
        return RLK_ERR_INVALID_VALUE;
    DeviceInfo dev;
    RLK_TRY(current_device(dev));
    CUtensorMap map_h, map_w;
    RLK_TRY(make_map(&map_h, hidden, H, N, H * 2, 64, rlk::kTileM));
    RLK_TRY(make_map(&map_w, weight_shard, H, V_local, H * 2, 64, rlk::kPairBRows));
    const float k = static_cast<float>(1.4426950408889634074 / temperature);
    RLK_CUDA(rlk::launch_fwd_partials(map_h, map_w, targets, active_mask, static_cast<int>(N),
                                      static_cast<int>(H), static_cast<int>(V_local),
                                      vocab_start, k, reinterpret_cast<float2*>(partials_out),
                                      target_logit_out, device_error_word, dev.sms, stream));
    return RLK_OK;
}

rlk_status_t rlk_linear_logp_merge(const float* partials, int64_t num_partials,
                                   const float* target_logit, const int64_t* targets,
                                   const uint8_t* active_mask, int64_t N, int64_t V,
                                   double temperature, float* logp_out, float* lse_out,
                                   uint32_t* device_error_word, cudaStream_t stream) {
    if (N < 0 || N > kMaxDim || V < 1 || V > kMaxDim) return RLK_ERR_INVALID_VALUE;
    if (!(std::isfinite(temperature) && temperature > 0.0)) return RLK_ERR_INVALID_VALUE;
    if (num_partials < 1 || num_partials > (int64_t(1) << 24)) return RLK_ERR_INVALID_VALUE;
    if (N == 0) return RLK_OK;
    if (partials == nullptr || target_logit == nullptr || targets == nullptr || logp_out == nullptr)
        return RLK_ERR_INVALID_VALUE;
    if (!aligned(partials, 8)) return RLK_ERR_INVALID_VALUE;
    DeviceInfo dev;
    RLK_TRY(current_device(dev));
    const float k = static_cast<float>(1.4426950408889634074 / temperature);
    RLK_CUDA(rlk::launch_fwd_merge(reinterpret_cast<const float2*>(partials),
                                   static_cast<int>(num_partials), target_logit, targets,
                                   active_mask, static_cast<int>(N), static_cast<int>(V), k,
                                   logp_out, lse_out, device_error_word, stream));
    return RLK_OK;
}

rlk_status_t rlk_logp_from_logits(const void* logits, int32_t dtype, int64_t N, int64_t V,
                                  int64_t row_stride, const int64_t* rows, int64_t M,
                                  const int64_t* targets, const uint8_t* active_mask,
                                  double temperature, float* logp_out, float* lse_out,
                                  uint32_t* device_error_word, cudaStream_t stream) {
    if (dtype != RLK_DTYPE_F32 && dtype != RLK_DTYPE_BF16) return RLK_ERR_UNSUPPORTED;
    if (N < 0 || N > kMaxDim || V < 1 || V > kMaxDim || row_stride < V) return RLK_ERR_INVALID_VALUE;
    if (!(std::isfinite(temperature) && temperature > 0.0)) return RLK_ERR_INVALID_VALUE;
    if (rows == nullptr) M = N;
    if (M < 0 || M > kMaxDim) return RLK_ERR_INVALID_VALUE;
    if (M == 0) return RLK_OK;
    if (logits == nullptr || targets == nullptr || logp_out == nullptr) return RLK_ERR_INVALID_VALUE;
    const size_t esize = dtype == RLK_DTYPE_F32 ? 4 : 2;
    if (!aligned(logits, esize)) return RLK_ERR_INVALID_VALUE;
    DeviceInfo dev;
    RLK_TRY(current_device(dev));
    const bool vec_ok = aligned(logits, 16) && (static_cast<size_t>(row_stride) * esize) % 16 == 0;
    const float k = static_cast<float>(1.4426950408889634074 / temperature);
    RLK_CUDA(rlk::launch_logp_from_logits(logits, dtype == RLK_DTYPE_BF16, row_stride, N,
                                          static_cast<int>(V), rows, static_cast<int>(M),
                                          targets, active_mask, k, vec_ok, logp_out, lse_out,
                                          device_error_word, stream));
    return RLK_OK;
}

size_t rlk_grpo_clip_loss_workspace_bytes(int64_t N) {
    if (N < 0) return 0;
    return align_up(rlk::loss_blocks(N) * sizeof(rlk::LossPartial), 256) + 256;
}

rlk_status_t rlk_grpo_clip_loss(const float* logp_new, const float* logp_old,
                                const float* advantages, const uint8_t* active_mask, int64_t N,
                                double eps_low, double eps_high, double loss_scale,
                                float* grad_out, rlk_grpo_result_t* result_dev, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
    if (N < 0 || N > (int64_t(1) << 40)) return RLK_ERR_INVALID_VALUE;
    if (!(std::isfinite(eps_low) && eps_low >= 0.0 && eps_low < 1.0)) return RLK_ERR_INVALID_VALUE;
    if (!(std::isfinite(eps_high) && eps_high >= 0.0)) return RLK_ERR_INVALID_VALUE;
    if (!(std::isfinite(loss_scale) && loss_scale > 0.0)) return RLK_ERR_INVALID_VALUE;
    if (result_dev == nullptr) return RLK_ERR_INVALID_VALUE;
    if (N > 0 && (logp_new == nullptr || logp_old == nullptr || advantages == nullptr ||
                  grad_out == nullptr))
        return RLK_ERR_INVALID_VALUE;
    if (workspace == nullptr || !aligned(workspace, 256) ||
        workspace_bytes < rlk_grpo_clip_loss_workspace_bytes(N))
        return RLK_ERR_WORKSPACE;
    DeviceInfo dev;
    RLK_TRY(current_device(dev));
    const bool vec_ok = aligned(logp_new, 16) && aligned(logp_old, 16) &&
                        aligned(advantages, 16) && aligned(grad_out, 16) &&
                        (active_mask == nullptr || aligned(active_mask, 4));
    RLK_CUDA(rlk::launch_grpo_loss(logp_new, logp_old, advantages, active_mask, N, eps_low,
                                   eps_high, loss_scale, grad_out, result_dev, workspace, vec_ok,
                                   stream));
    return RLK_OK;
}

size_t rlk_dlogp_audit_ext_workspace_bytes(int64_t N) {
    if (N < 0) return 0;
    return rlk::audit_ext_workspace(N);
}

rlk_status_t rlk_dlogp_audit_ext(const float* logp_new, const float* logp_old,
                                 const uint8_t* active_mask, int64_t N,
                                 const int64_t* seq_offsets, int64_t num_seqs, double clip_eps,
                                 rlk_audit_ext_t* result_dev, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream) {
    if (N < 0) return RLK_ERR_INVALID_VALUE;
    if (N > RLK_AUDIT_EXT_MAX_N) return RLK_ERR_UNSUPPORTED;   // 32-bit select counts
    if (result_dev == nullptr) return RLK_ERR_INVALID_VALUE;
    if (N > 0 && (logp_new == nullptr || logp_old == nullptr)) return RLK_ERR_INVALID_VALUE;
    if (!(std::isfinite(clip_eps) && clip_eps >= 0.0)) return RLK_ERR_INVALID_VALUE;
    if (seq_offsets != nullptr && num_seqs < 1) return RLK_ERR_INVALID_VALUE;
    if (workspace == nullptr || !aligned(workspace, 256) ||
        workspace_bytes < rlk_dlogp_audit_ext_workspace_bytes(N))
        return RLK_ERR_WORKSPACE;
    DeviceInfo dev;
    RLK_TRY(current_device(dev));
    const bool vec_ok = aligned(logp_new, 16) && aligned(logp_old, 16) &&
                        (active_mask == nullptr || aligned(active_mask, 4));
    RLK_CUDA(rlk::launch_audit_ext(logp_new, logp_old, active_mask, N, seq_offsets,
                                   seq_offsets == nullptr ? 0 : num_seqs,
                                   static_cast<float>(clip_eps), result_dev, workspace, vec_ok,
                                   dev.sms, stream));
    return RLK_OK;
}

rlk_status_t rlk_dlogp_audit_noalloc(const float* logp_new, const float* logp_old,
                                     const uint8_t* active_mask, int64_t N,
                                     rlk_audit_result_t* result_dev, cudaStream_t stream) {
    if (N < 0) return RLK_ERR_INVALID_VALUE;
    if (N > RLK_AUDIT_NOALLOC_MAX_N) return RLK_ERR_UNSUPPORTED;
    if (result_dev == nullptr) return RLK_ERR_INVALID_VALUE;
    if (N > 0 && (logp_new == nullptr || logp_old == nullptr)) return RLK_ERR_INVALID_VALUE;
    DeviceInfo dev;
    RLK_TRY(current_device(dev));
    void* scratch = nullptr;
    RLK_CUDA(rlk::audit_noalloc_scratch(&scratch));
    const bool vec_ok = aligned(logp_new, 16) && aligned(logp_old, 16) &&
                        (active_mask == nullptr || aligned(active_mask, 4));
    RLK_CUDA(rlk::launch_audit(logp_new, logp_old, active_mask, N, result_dev, scratch, vec_ok,
                               stream));
    return RLK_OK;
}

#define RLK_STR2(x) #x
#define RLK_STR(x) RLK_STR2(x)

const char* rlk_contract_string(void) {
    return "rlk-gb300 linear_logp v1; arch=sm_103a; nvcc=" RLK_STR(__CUDACC_VER_MAJOR__) "." RLK_STR(
        __CUDACC_VER_MINOR__) "; inputs=bf16; accum=fp32 (tcgen05 kind::f16, TMEM); "
                              "tiles: 256x256x64 on CTA pairs (cta_group::2) for the logp "
                              "and entropy GEMMs, 128x256x64 (cta_group::1) for the KL GEMMs; "
                              "no split-K; "
                              "fwd_vocab_chunk=1024 (merge ascending); bwd_vocab_chunk=32768; "
                              "masked batches: active rows compacted (ascending) before the "
                              "forward and backward GEMMs; "
                              "exp=ex2.approx.ftz, log=lg2.approx.ftz; k=fp32(log2(e)/T); "
                              "logits never rounded; logp/lse fp32; dS bf16 (target and "
                              "dominant-class terms fp32; entropy and KL: hi and lo bf16 "
                              "planes); "
                              "dh/dW rounded once to bf16 (RNE); no float atomics; "
                              "audit: 4096-element slices dealt round-robin to min(slices, 608) "
                              "blocks, fixed trees, float-pair (two-sum) partials; "
                              "data-parallel dW: fp32 partials merged in rank order, one "
                              "rounding";
}

const char* rlk_status_string(rlk_status_t status) {
    switch (status) {
        case RLK_OK: return "RLK_OK";
        case RLK_ERR_INVALID_VALUE: return "RLK_ERR_INVALID_VALUE";
        case RLK_ERR_UNSUPPORTED: return "RLK_ERR_UNSUPPORTED";
        case RLK_ERR_WORKSPACE: return "RLK_ERR_WORKSPACE";
        case RLK_ERR_LAUNCH: return "RLK_ERR_LAUNCH";
    }
    return "RLK_ERR_UNKNOWN";
}

}  // extern "C"
