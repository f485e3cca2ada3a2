// gemm.cuh -- persistent, warp-specialised bf16 GEMM mainloop for sm_103a.
//
//   warp 0      : TMA producer (one elected lane) filling a ring of
//                 shared-memory stages (A 128x64, B 256x64 or, for CTA
//                 pairs, its 128x64 half; 128-byte swizzle)
//   warp 1      : TMEM allocator and MMA issuer (one elected lane):
//                 tcgen05.mma.kind::f16, K=16, fp32 accumulators in TMEM,
//                 two 256-column buffers so the epilogue of tile i overlaps
//                 the MMAs of tile i+1
//   warps 2..   : epilogue (4 warps, or 8 for paired-tile policies), one
//                 thread per accumulator row (TMEM lane) and column half,
//                 reading 32-column slices with tcgen05.ld
//
// Two MMA shapes.  cta_group::1: one CTA, M=128 N=256.  CTA pairs
// (policies with kCtaPair): a cluster of two CTAs computes a 256x256 tile
// with tcgen05.mma.cta_group::2 M=256 N=256 -- each CTA loads 128 rows of A
// and 128 rows of B into its own ring (at the same offsets), the even CTA
// issues the MMAs, which read B from both CTAs, and each CTA's TMEM receives
// its 128 rows of the accumulator.  Per FLOP each SM then moves a third
// less operand data from L2 into shared memory and reads a third less from
// it.  Both CTAs' copies complete on the even CTA's "full" barrier, whose
// producer announces the bytes of both (a local arrive: a cluster-scope
// release on every stage would fence the producer and starve the MMAs); the
// even CTA's commits release the stage and signal "TMEM full" in both CTAs;
// both CTAs' epilogue warps arrive on the even CTA's "TMEM empty" barrier.
//
// The policy P decides the operands' majorness, the work units (a unit is a
// run of tiles that shares one epilogue state), tile coordinates, the K
// extent and the epilogue.  Every unit is processed start to finish by one
// CTA; units are dealt out round-robin (unit = blockIdx.x + i * gridDim.x).
// Nothing about the arithmetic of a tile depends on the grid: the K loop
// always runs in ascending 16-wide steps and never splits K.
//
// Waits are bounded (wall-clock timeout plus a shared abort flag).  A wait
// that gives up records RLK_DEVERR_WAIT_TIMEOUT, tells the other roles to
// stop, waits (bounded) for its own copies and MMAs in flight, and the CTA
// always frees its TMEM before it exits.
#pragma once

#include "ptx.cuh"
#include "rlk_internal.h"

namespace rlk {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kPairM = 2 * kBM;                    // rows of a CTA pair's tile
static_assert(kPairM == kUnitM, "the pair tile is the policies' unit");
constexpr int kStages = 4;                         // single CTA: 48 KiB stages
constexpr int kPairStages = 6;                     // CTA pair: 32 KiB stages
constexpr uint32_t kAStageBytes = kBM * kBK * 2;   // 16 KiB
constexpr uint32_t kBStageBytes = kBN * kBK * 2;   // 32 KiB
constexpr uint32_t kStageBytes = kAStageBytes + kBStageBytes;
constexpr uint32_t kTmemCols = 2 * kBN;            // two fp32 accumulators
constexpr int kGemmThreads = 192;
constexpr uint32_t kBarrierBytes = 256;
constexpr uint32_t kGemmSmemBytes = kStages * kStageBytes + kBarrierBytes + 1024;  // + align slack

// Ring geometry of a policy: stage count and bytes of each operand per stage.
template <bool PAIR>
struct RingShape {
    static constexpr int stages = PAIR ? kPairStages : kStages;
    static constexpr int b_rows = PAIR ? kBN / 2 : kBN;
    static constexpr uint32_t a_bytes = kAStageBytes;
    static constexpr uint32_t b_bytes = static_cast<uint32_t>(b_rows) * kBK * 2;
    static constexpr uint32_t stage_bytes = a_bytes + b_bytes;
    static constexpr uint32_t smem_bytes = stages * stage_bytes + kBarrierBytes + 1024;
};
static_assert(RingShape<true>::smem_bytes <= 227 * 1024, "CTA-pair ring exceeds shared memory");
constexpr uint64_t kWaitTimeoutNs = 4000000000ull;  // 4 s for one wait: far above any real wait
constexpr uint64_t kDrainTimeoutNs = 200000000ull;

// One TMA stage of an operand with `ROWS` rows along M (or N) and kBK along K.
//  K-major  : one box {64 (K), ROWS}; rows are 128 B apart, 8-row groups 1 KiB.
//  MN-major : ROWS/64 boxes {64 (MN), 64 (K)} of 8 KiB each; within a box the
//             64 K rows are 128 B apart.
template <bool MN_MAJOR, int ROWS>
__device__ __forceinline__ void load_operand(uint8_t* dst, const CUtensorMap* map, uint64_t* bar,
                                             int mn0, int k0) {
    if constexpr (!MN_MAJOR) {
        tma_load_2d(dst, map, bar, k0, mn0);
    } else {
#pragma unroll
        for (int i = 0; i < ROWS / 64; ++i) tma_load_2d(dst + i * 8192, map, bar, mn0 + 64 * i, k0);
    }
}

// Descriptor of the kk-th 16-wide K slice of a stage.
//  K-major  : the slice starts 32 B into each 128 B row (SBO = 1 KiB between
//             8-row groups; LBO unused by the 128 B swizzle).
//  MN-major : the slice is 16 K rows = two 1 KiB groups further on
//             (SBO = 1 KiB between 8-row K groups, LBO = 8 KiB between
//             64-element MN blocks).
template <bool MN_MAJOR>
__device__ __forceinline__ uint64_t operand_desc(uint32_t stage_addr, int kk) {
    if constexpr (!MN_MAJOR) {
        return smem_desc_sw128(stage_addr + kk * 32, 16, 1024);
    } else {
        return smem_desc_sw128(stage_addr + kk * 2048, 8192, 1024);
    }
}

// The same for one CTA of a pair: the copies complete on the even CTA's barrier
// (bar: shared::cluster address).
template <bool MN_MAJOR, int ROWS>
__device__ __forceinline__ void load_operand_pair(uint8_t* dst, const CUtensorMap* map,
                                                  uint32_t bar, int mn0, int k0) {
    if constexpr (!MN_MAJOR) {
        tma_load_2d_pair(dst, map, bar, k0, mn0);
    } else {
#pragma unroll
        for (int i = 0; i < ROWS / 64; ++i)
            tma_load_2d_pair(dst + i * 8192, map, bar, mn0 + 64 * i, k0);
    }
}

template <int ROWS>
__device__ __forceinline__ void load_operand_pair_rt(bool mn_major, uint8_t* dst,
                                                     const CUtensorMap* map, uint32_t bar,
                                                     int mn0, int k0) {
    if (mn_major)
        load_operand_pair<true, ROWS>(dst, map, bar, mn0, k0);
    else
        load_operand_pair<false, ROWS>(dst, map, bar, mn0, k0);
}

// Runtime-majorness variants for policies that mix operand layouts per unit.
template <int ROWS>
__device__ __forceinline__ void load_operand_rt(bool mn_major, uint8_t* dst, const CUtensorMap* map,
                                                uint64_t* bar, int mn0, int k0) {
    if (mn_major)
        load_operand<true, ROWS>(dst, map, bar, mn0, k0);
    else
        load_operand<false, ROWS>(dst, map, bar, mn0, k0);
}

__device__ __forceinline__ uint64_t operand_desc_rt(bool mn_major, uint32_t stage_addr, int kk) {
    return mn_major ? operand_desc<true>(stage_addr, kk) : operand_desc<false>(stage_addr, kk);
}

// The policy interface the mainloop relies on:
//   struct Maps                          tensor maps (kernel parameter)
//   a_map(maps, u), b_map(maps, u)        maps of unit u's operands
//   a_mn(u), b_mn(u)                      operand majorness of unit u
//   num_units(), tiles_in_unit(u), k_blocks(u), coords(u, q, ...)
//   EpiState, epi_begin / epi_tile / epi_end
//   kPairTiles                            false: one epilogue call per tile
//   kKRemap, k_remap(kb, nkb, a_mn, a_k, b_mn, b_k)
//                                         true: the coordinates of K block kb
//                                         (of nkb) are the policy's, not the
//                                         plain ascending walk along K
//   kCtaPair                              true: units are 256-row tiles of a
//                                         CTA pair; coords() gives the tile's
//                                         origin, the mainloop adds the CTA's
//                                         128-row offset to both operands, and
//                                         the epilogue's row runs over 0..255
// With kPairTiles the tiles of a unit come in pairs (2i, 2i+1) that may use
// different operands (tile_a_map / tile_b_map / tile_k_blocks(u, q)); the
// epilogue sees both accumulators at once (epi_pair, after the odd tile) and
// releases the two TMEM buffers together.  Units then hold an even number of
// tiles, so a pair always occupies buffers 0 and 1.  Paired tiles also run on
// CTA pairs: each CTA's epilogue warps take its 128 rows of both accumulators and
// arrive on the leader's barriers.  Pair policies may set
// kEpiWarps = 8: two warps per TMEM lane quarter, each given half of the
// tile's columns (epi_begin / epi_pair / epi_end take the half), so that the
// epilogue, which the MMA waits for, takes half as long.  epi_pair also gets the
// kernel's tensor maps and, for a policy with kEpiSmemPerWarp > 0, this warp's
// slot of that many bytes of shared memory (after the ring), e.g. to stage a tile
// for a TMA store; such a warp waits for its bulk stores before the CTA exits.
// TwoMaps serves the single-role policies.
struct TwoMaps {
    CUtensorMap a, b;
};

// Mixin for policies whose every unit has the same operand layouts and maps.
template <bool AMN, bool BMN>
struct SingleRole {
    using Maps = TwoMaps;
    static constexpr bool kPairTiles = false;
    static constexpr bool kKRemap = false;
    static constexpr bool kCtaPair = false;
    static constexpr int kEpiWarps = 4;
    static constexpr int kEpiSmemPerWarp = 0;
    static constexpr bool kAMn = AMN;
    static constexpr bool kBMn = BMN;
    __device__ static void prefetch(const Maps& m) {
        prefetch_tensormap(&m.a);
        prefetch_tensormap(&m.b);
    }
    __device__ static const CUtensorMap* a_map(const Maps& m, int) { return &m.a; }
    __device__ static const CUtensorMap* b_map(const Maps& m, int) { return &m.b; }
    __device__ static bool a_mn(int) { return AMN; }
    __device__ static bool b_mn(int) { return BMN; }
};

// Grouped raster of a rows x cols grid of work units: units are visited
// group by group, a group being `group` consecutive rows (the last group may
// be shorter) times every column, with the row index running fastest inside a
// group.  Concurrent CTAs then share one group's rows (kept in L2) while the
// column operand streams.  Only the visiting order changes, never a unit's
// arithmetic.
__device__ __forceinline__ void grouped_unit(int u, int rows, int cols, int group, int& r,
                                             int& c) {
    const int full = rows / group;
    const int per_group = group * cols;
    const int g = u / per_group;
    if (g < full) {
        const int l = u - g * per_group;
        c = l / group;
        r = g * group + (l - c * group);
    } else {
        const int gr = rows - full * group;
        const int l = u - full * per_group;
        c = l / gr;
        r = full * group + (l - c * gr);
    }
}

// x[i] for a runtime i in [0, 32) through a fixed 5-level select tree, so
// that the 32 values stay in registers.
__device__ __forceinline__ float select32(const float (&x)[32], int i) {
    float a[16], b[8], c[4], d[2];
#pragma unroll
    for (int j = 0; j < 16; ++j) a[j] = (i & 16) ? x[j + 16] : x[j];
#pragma unroll
    for (int j = 0; j < 8; ++j) b[j] = (i & 8) ? a[j + 8] : a[j];
#pragma unroll
    for (int j = 0; j < 4; ++j) c[j] = (i & 4) ? b[j + 4] : b[j];
#pragma unroll
    for (int j = 0; j < 2; ++j) d[j] = (i & 2) ? c[j + 2] : c[j];
    return (i & 1) ? d[1] : d[0];
}

__device__ __forceinline__ void report_error(uint32_t* err, uint32_t bits) {
    if (err != nullptr) atomicOr(err, bits);
}

// threads of a launch: the TMA warp, the MMA warp and the epilogue warps
template <class P>
constexpr int gemm_threads() {
    return 64 + 32 * P::kEpiWarps;
}

template <class P>
__host__ __device__ constexpr uint32_t gemm_smem_bytes() {
    return RingShape<P::kCtaPair>::smem_bytes +
           static_cast<uint32_t>(P::kEpiWarps * P::kEpiSmemPerWarp);
}

// Programmatic dependent launch between two GEMM launches that share no data:
// kPdlTrigger lets the next launch start on SMs as this grid's CTAs finish;
// kPdlOverlap launches a GEMM that does not wait for the previous grid to start,
// only to end (it reads and writes nothing that grid touches).
constexpr unsigned kPdlTrigger = 1u;
constexpr unsigned kPdlOverlap = 2u;

template <class P>
__global__ void __launch_bounds__(64 + 32 * P::kEpiWarps, 1)
    gemm_persistent_kernel(const __grid_constant__ typename P::Maps maps, const P p,
                           uint32_t* err, unsigned pdl) {
    constexpr bool PAIR = P::kCtaPair;
    using Ring = RingShape<PAIR>;
    constexpr int S = Ring::stages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* a_stages = smem;
    uint8_t* b_stages = smem + S * Ring::a_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * Ring::stage_bytes);
    uint8_t* epi_smem = smem + S * Ring::stage_bytes + kBarrierBytes;   // [kEpiWarps] slots
    static_assert(gemm_smem_bytes<P>() <= 227 * 1024, "shared memory of the launch");
    uint64_t* full = bars;                    // [S] TMA -> MMA (pair: the even CTA's counts both CTAs' bytes)
    uint64_t* empty = bars + S;               // [S] MMA -> TMA
    uint64_t* tmem_full = bars + 2 * S;       // [2] MMA -> epilogue
    uint64_t* tmem_empty = tmem_full + 2;     // [2] epilogue -> MMA (pair: both CTAs' warps)
    uint64_t* drain = tmem_empty + 2;         // [1] MMA self-drain
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    volatile int* never = abort_flag + 1;     // stays 0: drain waits ignore the abort flag

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // the unit stream of this CTA (pair: of its cluster) and this CTA's row offset in it
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const int wg = PAIR ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
    const int num_wg = PAIR ? static_cast<int>(num_clusters_x()) : static_cast<int>(gridDim.x);
    const int half_off = static_cast<int>(rank) * kBM;

    if (warp == 0 && lane == 0) {
        P::prefetch(maps);
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tmem_full[b], 1);
            mbar_init(&tmem_empty[b], (PAIR ? 2 : 1) * P::kEpiWarps);   // one arrival per epilogue warp
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *never = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(tmem_holder, kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_holder, kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();       // the peer's barriers exist before any remote arrival
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // every CTA is resident: the next launch in the stream may be scheduled onto the
    // SMs that this grid's CTAs leave
    if (pdl & kPdlTrigger) asm volatile("griddepcontrol.launch_dependents;");

    const int units = p.num_units();

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_parity = 0;
            bool ok = true;
            for (int u = wg; ok && u < units; u += num_wg) {
                const int nt = p.tiles_in_unit(u);
                const int kblocks = p.k_blocks(u);
                const bool amn = p.a_mn(u), bmn = p.b_mn(u);
                const CUtensorMap* ma = p.a_map(maps, u);
                const CUtensorMap* mb = p.b_map(maps, u);
                for (int q = 0; ok && q < nt; ++q) {
                    int a_mn, a_k, b_mn, b_k;
                    p.coords(u, q, a_mn, a_k, b_mn, b_k);
                    const CUtensorMap* qa = ma;
                    const CUtensorMap* qb = mb;
                    int qk = kblocks;
                    if constexpr (P::kPairTiles) {
                        qa = p.tile_a_map(maps, u, q);
                        qb = p.tile_b_map(maps, u, q);
                        qk = p.tile_k_blocks(u, q);
                    }
                    for (int kb = 0; kb < qk; ++kb) {
                        const bool got = PAIR
                            ? mbar_wait_cluster(&empty[stage], phase ^ 1u, abort_flag, kWaitTimeoutNs)
                            : mbar_wait(&empty[stage], phase ^ 1u, abort_flag, kWaitTimeoutNs);
                        if (!got) {
                            ok = false;
                            break;
                        }
                        int am = a_mn, ak = a_k + kb * kBK, bm = b_mn, bk = b_k + kb * kBK;
                        if constexpr (P::kKRemap) p.k_remap(kb, qk, am, ak, bm, bk);
                        if constexpr (PAIR) {
                            // the even CTA's barrier counts both CTAs' bytes: its producer
                            // announces them with a local arrive, the odd CTA's copies only
                            // complete on it (no fence on this path)
                            const uint32_t lf = mapa_shared(smem_u32(&full[stage]), 0);
                            if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * Ring::stage_bytes);
                            load_operand_pair_rt<kBM>(amn, a_stages + stage * Ring::a_bytes, qa, lf,
                                                      am + half_off, ak);
                            load_operand_pair_rt<Ring::b_rows>(bmn, b_stages + stage * Ring::b_bytes,
                                                               qb, lf, bm + half_off, bk);
                        } else {
                            mbar_arrive_expect_tx(&full[stage], Ring::stage_bytes);
                            load_operand_rt<kBM>(amn, a_stages + stage * Ring::a_bytes, qa,
                                                 &full[stage], am, ak);
                            load_operand_rt<kBN>(bmn, b_stages + stage * Ring::b_bytes, qb,
                                                 &full[stage], bm, bk);
                        }
                        issued_mask |= 1u << stage;
                        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                        if (++stage == S) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            if (!ok) {
                report_error(err, RLK_DEVERR_WAIT_TIMEOUT);
                *abort_flag = 1;
            }
            // let every copy this thread started land before the CTA can exit (pair: the
            // even CTA's MMAs release a stage only after reading it, so a released stage
            // has landed)
            for (int s = 0; s < S; ++s)
                if (issued_mask & (1u << s)) {
                    if constexpr (PAIR)
                        mbar_wait_cluster(&empty[s], (issued_parity >> s) & 1u, never, kDrainTimeoutNs);
                    else
                        mbar_wait(&full[s], (issued_parity >> s) & 1u, never, kDrainTimeoutNs);
                }
        }
    } else if (warp == 1) {
        if (lane == 0 && (!PAIR || rank == 0)) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t tile_i = 0;
            bool ok = true;
            for (int u = wg; ok && u < units; u += num_wg) {
                const int nt = p.tiles_in_unit(u);
                const int kblocks = p.k_blocks(u);
                const bool amn = p.a_mn(u), bmn = p.b_mn(u);
                const uint32_t idesc = idesc_bf16_f32(PAIR ? kPairM : kBM, kBN, amn, bmn);
                for (int q = 0; ok && q < nt; ++q, ++tile_i) {
                    const uint32_t buf = tile_i & 1u;
                    const uint32_t use = tile_i >> 1;
                    const bool got = PAIR
                        ? mbar_wait_cluster(&tmem_empty[buf], (use & 1u) ^ 1u, abort_flag, kWaitTimeoutNs)
                        : mbar_wait(&tmem_empty[buf], (use & 1u) ^ 1u, abort_flag, kWaitTimeoutNs);
                    if (!got) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * kBN;
                    int qk = kblocks;
                    if constexpr (P::kPairTiles) qk = p.tile_k_blocks(u, q);
                    for (int kb = 0; kb < qk; ++kb) {
                        const bool landed = PAIR
                            ? mbar_wait_cluster(&full[stage], phase, abort_flag, kWaitTimeoutNs)
                            : mbar_wait(&full[stage], phase, abort_flag, kWaitTimeoutNs);
                        if (!landed) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_addr = smem_u32(a_stages + stage * Ring::a_bytes);
                        const uint32_t b_addr = smem_u32(b_stages + stage * Ring::b_bytes);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {
                            if constexpr (PAIR)
                                mma_bf16_ss_pair(d_tmem, operand_desc_rt(amn, a_addr, kk),
                                                 operand_desc_rt(bmn, b_addr, kk), idesc,
                                                 (kb > 0 || kk > 0) ? 1u : 0u);
                            else
                                mma_bf16_ss(d_tmem, operand_desc_rt(amn, a_addr, kk),
                                            operand_desc_rt(bmn, b_addr, kk), idesc,
                                            (kb > 0 || kk > 0) ? 1u : 0u);
                        }
                        if constexpr (PAIR)
                            mma_commit_pair(&empty[stage], 3);
                        else
                            mma_commit(&empty[stage]);
                        if (++stage == S) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (ok) {
                        if constexpr (PAIR)
                            mma_commit_pair(&tmem_full[buf], 3);
                        else
                            mma_commit(&tmem_full[buf]);
                    }
                }
            }
            if (!ok) {
                report_error(err, RLK_DEVERR_WAIT_TIMEOUT);
                *abort_flag = 1;
            }
            // every MMA issued by this thread completes before TMEM is freed
            if constexpr (PAIR)
                mma_commit_pair(drain, 1);
            else
                mma_commit(drain);
            mbar_wait(drain, 0, never, kDrainTimeoutNs);
        }
    } else {
        const int quarter = warp & 3;         // TMEM lanes this warp may access
        const int half = (warp - 2) >> 2;     // column half (0 unless kEpiWarps = 8)
        const int row = quarter * 32 + lane;  // this thread's accumulator row in the CTA
        const int prow = half_off + row;      // ... in the unit's tile (pair: 0..255)
        const uint32_t taddr_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
        uint32_t tile_i = 0;
        bool ok = true;
        for (int u = wg; ok && u < units; u += num_wg) {
            typename P::EpiState st;
            if constexpr (P::kPairTiles)
                p.epi_begin(u, prow, half, st);
            else
                p.epi_begin(u, prow, st);
            const int nt = p.tiles_in_unit(u);
            for (int q = 0; q < nt; ++q, ++tile_i) {
                const uint32_t buf = tile_i & 1u;
                const uint32_t use = tile_i >> 1;
                int got = 1;
                if (lane == 0)
                    got = PAIR ? mbar_wait_cluster(&tmem_full[buf], use & 1u, abort_flag, kWaitTimeoutNs)
                               : mbar_wait(&tmem_full[buf], use & 1u, abort_flag, kWaitTimeoutNs);
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) {
                    ok = false;
                    break;
                }
                if constexpr (P::kPairTiles) {
                    if ((q & 1) == 0) continue;       // hold the even tile's buffer
                    tc_fence_after();
                    p.epi_pair(maps, u, q, prow, half, taddr_row + (buf ^ 1u) * kBN,
                               taddr_row + buf * kBN, st,
                               epi_smem + (warp - 2) * P::kEpiSmemPerWarp);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (PAIR) {
                            mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_empty[buf ^ 1u]), 0));
                            mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_empty[buf]), 0));
                        } else {
                            mbar_arrive(&tmem_empty[buf ^ 1u]);
                            mbar_arrive(&tmem_empty[buf]);
                        }
                    }
                } else {
                    tc_fence_after();
                    p.epi_tile(u, q, prow, taddr_row + buf * kBN, st);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (PAIR)
                            mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_empty[buf]), 0));
                        else
                            mbar_arrive(&tmem_empty[buf]);
                    }
                }
            }
            if (!ok) break;
            if constexpr (P::kPairTiles)
                p.epi_end(u, prow, half, st);
            else
                p.epi_end(u, prow, st);
        }
        if (!ok && lane == 0) {
            report_error(err, RLK_DEVERR_WAIT_TIMEOUT);
            *abort_flag = 1;
        }
        if constexpr (P::kEpiSmemPerWarp > 0) {
            if (lane == 0) bulk_wait_group0();   // this warp's bulk stores are done
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();       // the peer is done with this CTA's ring and TMEM
    if (warp == 1) {
        tc_fence_after();
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem_base, kTmemCols);
        else
            tmem_dealloc(tmem_base, kTmemCols);
    }
    // a launch that overlapped the previous grid ends only after that grid has, so
    // that whatever follows in the stream sees both complete
    if (pdl & kPdlOverlap) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launch of a persistent GEMM: one CTA (pair: one cluster of two) per SM (pair: per
// two SMs) up to the number of units.
template <class P>
cudaError_t launch_persistent(const typename P::Maps& maps, const P& p, long long units,
                              int num_sms, uint32_t* err, cudaStream_t stream,
                              unsigned pdl = 0) {
    auto kern = gemm_persistent_kernel<P>;
    constexpr uint32_t smem = gemm_smem_bytes<P>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const long long slots = P::kCtaPair ? num_sms / 2 : num_sms;
    const long long groups = units < slots ? units : slots;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((P::kCtaPair ? 2 : 1) * (groups > 0 ? groups : 1)));
    cfg.blockDim = dim3(gemm_threads<P>());
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (P::kCtaPair) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 2;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl & kPdlOverlap) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, maps, p, err, pdl);
}

}  // namespace rlk
