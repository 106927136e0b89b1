// gemm_pair_kernel.cuh -- the NVFP4 grouped GEMM on CTA pairs (sm_103a).
//
// A cluster of two CTAs on the two SMs of one TPC computes 256 x BN output
// tiles with tcgen05.mma.cta_group::2 (M = 256): each CTA stages its own 128
// rows of A and its own BN/2 rows of B, and the even CTA's single MMA thread
// drives the tensor cores of both SMs, each reading A from its own shared
// memory and B from both.  Per SM and per 128 x BN x 64 product that is
// 16 KB + BN*16 B of operands read from shared memory instead of
// 16 KB + BN*32 B with one CTA, and half the B bytes brought in through L2.
//
// Roles (warps, both CTAs unless noted):
//   0-3  epilogue: this CTA's 128 accumulator rows (its own tensor memory)
//        -> FP16 -> swizzled staging -> TMA tensor stores; hands the
//        accumulator back by arriving on the even CTA's acc_empty;
//   4    MMA issuer (even CTA, one thread); allocates / frees the pair's
//        tensor memory in both CTAs;
//   5    scale copier (even CTA, one thread): tcgen05.cp.cta_group::2 of the
//        stage's scale atoms into both CTAs' tensor memory;
//   6-9  loaders, one TMA thread and one operation per stage each: this CTA's
//        A tile [128 x 128 B] and its half of the B tile [BN/2 x 128 B]
//        (on full[slot]), this CTA's A scale atoms and the scale atoms of the
//        whole B tile (on sf_full[slot]; every CTA's tensor memory holds the
//        B scales of all BN columns);
//   10   L2 prefetcher of this CTA's B half, paced by its B loader.
// Loads of both CTAs complete on the even CTA's full / sf_full barriers (TMA
// .cta_group::2), whose arrivals (the even CTA's loaders) expect the bytes of
// both CTAs; MMA completion is multicast to both CTAs' empty[slot] and
// acc_full barriers.
//
// The tile roles, descriptors and scale addressing follow kernelbot
// nvfp4-group-gemm submission 474067 (group_gemm_persistent_kernel,
// tcgen05_mma_nvfp4, tcgen05_cp_nvfp4), which runs one CTA per tile; the
// pairing, the cross-CTA barrier protocol and the bounded waits are this
// build's own.
//
// Every wait on an mbarrier is bounded as in gemm_kernel.cuh.  Both CTAs
// meet in a cluster barrier after their roles have drained (bounded), so no
// remote arrive, copy completion or operand read can reach a CTA that has
// exited.
#pragma once

#include "gemm_kernel.cuh"

namespace nvfp4 {

// Launches take KernelParams (gemm_kernel.cuh) with tmA: box {128, 128, 1}
// (this CTA's 128 rows), tmB: box {128, BN/2, 1}, tmSFA box {128, 4, 1},
// tmSFB box {128, 4, BN/128}; grid_m / tile_end count 256-row tiles.

template <int BN_, int STAGES_, int EPI_COLS_>
struct PairConfig {
    static constexpr int BN = BN_;
    static constexpr int BK = kChunkK;                     // one 128-byte chunk per row per stage
    static constexpr int kStages = STAGES_;
    static constexpr int kEpiCols = EPI_COLS_;
    static_assert(BN == 256, "pair tiles are 256 x 256");
    static_assert(kEpiCols == 32 || kEpiCols == 64, "epilogue chunk must be 32 or 64 columns");
    static constexpr int kPairBM = 2 * kBM;
    static constexpr int kMmas = BK / kMmaK;               // 4
    static constexpr int kSfRb = BN / 128;                 // scale row blocks of the B tile
    static constexpr int kABytes = kBM * BK / 2;           // 16 KiB
    static constexpr int kBBytes = (BN / 2) * BK / 2;      // this CTA's half
    static constexpr int kSfaBytes = kMmas * 512;
    static constexpr int kSfbBytes = kSfRb * kMmas * 512;
    static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1 KiB alignment");
    // bytes of one stage over both CTAs, as the even CTA's producers expect them
    static constexpr uint32_t kTx[4] = {2u * kABytes, 2u * kBBytes, 2u * kSfaBytes, 2u * kSfbBytes};
    static constexpr int kEpiBufBytes = 32 * kEpiCols * 2;
    static constexpr int kEpiOff = kStages * kStageBytes;
    static constexpr int kBarOff = kEpiOff + 4 * kEpiBufBytes;
    // full[S], empty[S], sf_ready[S], sf_full[S], acc_full, acc_empty, drain,
    // sf_drain
    static constexpr int kNumBars = 4 * kStages + 4;
    static constexpr int kSlotOff = kBarOff + 8 * kNumBars;  // tmem base, abort flag, B progress
    static constexpr int kSmemBytes = kSlotOff + 16 + 1024;
    static_assert(kSmemBytes <= kSmemLimit, "exceeds 227 KiB of shared memory");
    static_assert(kStages * kStageBytes >= 4 * (BN / 64) * 4096, "ring too small for the last tile's slabs");
    static constexpr int kMmaWarpP = 4;
    static constexpr int kSfWarpP = 5;
    static constexpr int kFirstLoader = 6;   // A, B, A scales, B scales
    static constexpr int kPrefetchWarp = 10;
    static constexpr int kThreads = 32 * (kPrefetchWarp + 1);
    static constexpr int kTmemCols = 512;
    static constexpr int kSfCol0 = BN;                     // one accumulator
    static constexpr int kSfSlotCols = 4 * kMmas * (1 + kSfRb);
    static_assert(kSfCol0 + kStages * kSfSlotCols <= kTmemCols, "tensor memory budget");
    static constexpr uint32_t sfa_col(int slot, int j) { return kSfCol0 + slot * kSfSlotCols + 4 * j; }
    static constexpr uint32_t sfb_col(int slot, int j, int h)
    {
        return kSfCol0 + slot * kSfSlotCols + 4 * kMmas + 4 * kSfRb * j + 4 * h;
    }
    // kind::mxf4nvf4 instruction descriptor as for one CTA, with M = 256
    static constexpr uint32_t kIdesc =
        (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kPairBM >> 7) << 27);
};

// bounded drain wait that reports whether the phase completed
__device__ __noinline__ bool wait_drain_ok(uint32_t bar, uint32_t parity, const WaitCtx &w)
{
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > w.timeout_ns) {
            atomicOr(w.err, kErrDrainTimeout);
            atomicCAS(w.err + 1, 0u, (blockIdx.x << 4) | kRoleDrain);
            return false;
        }
    }
    return true;
}

// One loader of one CTA of the pair: ROLE 0 this CTA's A rows, 1 this CTA's
// half of the B tile (both on full[slot]), 2 this CTA's A scale atoms, 3 the
// scale atoms of the whole B tile (both on sf_full[slot]).  Loads complete on
// the even CTA's barrier; only the even CTA's loaders arrive there (with the
// bytes of both CTAs).
template <class Cfg, int ROLE>
__device__ __forceinline__ void pair_loader(const KernelParams &kp, uint32_t base, uint32_t bar0,
                                            uint32_t rank, volatile uint32_t *b_progress,
                                            const WaitCtx &wctx)
{
    const GemmParams &p = kp.g;
    constexpr int S = Cfg::kStages;
    constexpr bool kSf = ROLE >= 2;
    constexpr uint32_t kOff = ROLE == 0   ? 0u
                              : ROLE == 1 ? (uint32_t)Cfg::kABytes
                              : ROLE == 2 ? (uint32_t)(Cfg::kABytes + Cfg::kBBytes)
                                          : (uint32_t)(Cfg::kABytes + Cfg::kBBytes + Cfg::kSfaBytes);
    auto done_bar = [&](int s) { return bar0 + 8u * ((kSf ? 3 * S : 0) + s); };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };

    const bool b_side = (ROLE == 1 || ROLE == 3);
    const uint64_t pol = b_side ? (p.b_policy == 1   ? ptx::policy_evict_first()
                                   : p.b_policy == 2 ? ptx::policy_evict_last()
                                                     : ptx::policy_evict_normal())
                                : ptx::policy_evict_last();
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
    uint32_t q = 0;
    uint32_t issued = 0, issued_parity = 0;
    bool ok = true;
    int g = 0;
    for (int t = pair; t < p.total_tiles && ok; t += npairs) {
        const TileCoord tc = tile_coord(p, t, g);
        const int nst = p.kchunks[tc.g];                    // one 256-K chunk per stage
        for (int it = 0; it < nst; ++it, ++q) {
            const int stage = (int)(q % S);
            const uint32_t phase = (q / S) & 1u;
            if (!wait_bounded(empty_bar(stage), phase ^ 1u, wctx, kRoleProducer)) {
                ok = false;
                break;
            }
            const bool drop = ROLE == 1 && p.debug_drop_stage && blockIdx.x == 0 && q == 0;
            if (!drop) {
                const uint32_t dst = base + stage * Cfg::kStageBytes + kOff;
                const uint32_t bar_leader = ptx::mapa_shared(done_bar(stage), 0);
                if (rank == 0)
                    ptx::mbar_arrive_expect_tx(done_bar(stage), Cfg::kTx[ROLE]);
                if (ROLE == 0)
                    ptx::tma_load_3d_pair(dst, &p.tmA[tc.g], 0, tc.bm * Cfg::kPairBM + (int)rank * kBM, it,
                                          bar_leader, pol);
                else if (ROLE == 1)
                    ptx::tma_load_3d_pair(dst, &p.tmB[tc.g], 0,
                                          tc.bn * Cfg::BN + (int)rank * (Cfg::BN / 2), it, bar_leader, pol);
                else if (ROLE == 2)
                    ptx::tma_load_3d_pair(dst, &kp.tmSFA[tc.g], 0, it * Cfg::kMmas, tc.bm * 2 + (int)rank,
                                          bar_leader, pol);
                else
                    ptx::tma_load_3d_pair(dst, &kp.tmSFB[tc.g], 0, it * Cfg::kMmas, tc.bn * Cfg::kSfRb,
                                          bar_leader, pol);
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            }
            if (ROLE == 1)
                *b_progress = q + 1;
        }
    }
    (void)ok;
    // Loads issued but not yet consumed still land in this CTA's shared
    // memory.  The even CTA waits for its own barriers' phases (they count
    // the bytes of both CTAs); the odd CTA cannot see those and waits instead
    // for the MMAs to release its slots, giving up at the first expiry.
    bool alive = true;
    for (int s = 0; s < S && alive; ++s) {
        if (!(issued & (1u << s)))
            continue;
        const uint32_t par = (issued_parity >> s) & 1u;
        alive = rank == 0 ? wait_drain_ok(done_bar(s), par, wctx)
                          : wait_drain_ok(empty_bar(s), par, wctx);
    }
}

// L2 prefetch of this CTA's B half and its own B scale block, up to
// `pf_stages` stages ahead of this CTA's B producer
template <class Cfg>
__device__ __forceinline__ void pair_prefetch(const KernelParams &kp, uint32_t rank,
                                              volatile uint32_t *b_progress, const WaitCtx &wctx)
{
    const GemmParams &p = kp.g;
    const uint64_t pol = p.b_policy == 1   ? ptx::policy_evict_first()
                         : p.b_policy == 2 ? ptx::policy_evict_last()
                                           : ptx::policy_evict_normal();
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
    uint32_t q = 0;
    int g = 0;
    for (int t = pair; t < p.total_tiles; t += npairs) {
        const TileCoord tc = tile_coord(p, t, g);
        const int nst = p.kchunks[tc.g];
        const int row0 = tc.bn * Cfg::BN + (int)rank * (Cfg::BN / 2);
        const int rb = tc.bn * Cfg::kSfRb;
        for (int it = 0; it < nst; ++it, ++q) {
            if (q >= *b_progress + (uint32_t)p.pf_stages) {
                const uint64_t t0 = ptx::globaltimer_ns();
                while (q >= *b_progress + (uint32_t)p.pf_stages) {
                    if (*wctx.abort || ptx::globaltimer_ns() - t0 > wctx.timeout_ns)
                        return;
                    __nanosleep(128);
                }
            }
            ptx::tma_prefetch_3d(&p.tmB[tc.g], 0, row0, it, pol);
            if (rank == 0)
                ptx::tma_prefetch_3d(&kp.tmSFB[tc.g], 0, it * Cfg::kMmas, rb, pol);
        }
    }
}

template <class Cfg, bool EPI_EX>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    nvfp4_group_gemm_pair_kernel(const __grid_constant__ KernelParams kp)
{
    const GemmParams &p = kp.g;
    constexpr int BN = Cfg::BN;
    constexpr int S = Cfg::kStages;
    constexpr int EC = Cfg::kEpiCols;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);

    const uint32_t bar0 = base + Cfg::kBarOff;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto sfr_bar = [&](int s) { return bar0 + 8u * (2 * S + s); };
    auto sffull_bar = [&](int s) { return bar0 + 8u * (3 * S + s); };
    const uint32_t accf_bar = bar0 + 8u * (4 * S);
    const uint32_t acce_bar = bar0 + 8u * (4 * S + 1);
    const uint32_t drain_bar = bar0 + 8u * (4 * S + 2);
    const uint32_t sf_drain_bar = bar0 + 8u * (4 * S + 3);
    const uint32_t tmem_slot = base + Cfg::kSlotOff;
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + Cfg::kSlotOff + 4);
    volatile uint32_t *b_progress = reinterpret_cast<volatile uint32_t *>(gbase + Cfg::kSlotOff + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full_bar(s), 2);     // the even CTA's A and B loaders
            ptx::mbar_init(empty_bar(s), 1);
            ptx::mbar_init(sfr_bar(s), 1);
            ptx::mbar_init(sffull_bar(s), 2);   // the even CTA's scale loaders
        }
        ptx::mbar_init(accf_bar, 1);
        ptx::mbar_init(acce_bar, 8);          // lane 0 of the 4 epilogue warps of both CTAs
        ptx::mbar_init(drain_bar, 1);
        ptx::mbar_init(sf_drain_bar, 1);
        *abort_flag = 0u;
        *b_progress = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == Cfg::kMmaWarpP) {
        ptx::tmem_alloc_pair(tmem_slot, Cfg::kTmemCols);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    __syncthreads();
    // both CTAs' barriers are initialised before either CTA signals the other
    ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem_base = ptx::ld_shared_u32(tmem_slot);
    // the A and B loads of an early_ab launch do not wait for the previous
    // kernel (the library's scale relayout, which reads neither)
    if (!(p.early_ab && (warp == Cfg::kFirstLoader || warp == Cfg::kFirstLoader + 1)))
        ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();

    const WaitCtx wctx{abort_flag, p.err, p.timeout_ns};
    const int total = p.total_tiles;
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);

    if (warp == Cfg::kPrefetchWarp) {
        if (lane == 0 && p.pf_stages > 0)
            pair_prefetch<Cfg>(kp, rank, b_progress, wctx);
    } else if (warp >= Cfg::kFirstLoader) {
        if (lane == 0) {
            switch (warp - Cfg::kFirstLoader) {
            case 0: pair_loader<Cfg, 0>(kp, base, bar0, rank, b_progress, wctx); break;
            case 1: pair_loader<Cfg, 1>(kp, base, bar0, rank, b_progress, wctx); break;
            case 2: pair_loader<Cfg, 2>(kp, base, bar0, rank, b_progress, wctx); break;
            default: pair_loader<Cfg, 3>(kp, base, bar0, rank, b_progress, wctx); break;
            }
        }
    } else if (warp == Cfg::kSfWarpP) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------- scale copies
            uint32_t q = 0;
            bool ok = true, issued_any = false;
            int g = 0;
            for (int t = pair; t < total && ok; t += npairs) {
                const TileCoord tc = tile_coord(p, t, g);
                const int nst = p.kchunks[tc.g];
                for (int it = 0; it < nst; ++it, ++q) {
                    const int stage = (int)(q % S);
                    if (!wait_bounded(sffull_bar(stage), (q / S) & 1u, wctx, kRoleSf)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t ssfa = base + stage * Cfg::kStageBytes + Cfg::kABytes + Cfg::kBBytes;
                    const uint32_t ssfb = ssfa + Cfg::kSfaBytes;
#pragma unroll
                    for (int j = 0; j < Cfg::kMmas; ++j) {
                        ptx::tc_cp_32x128b_warpx4_pair(tmem_base + Cfg::sfa_col(stage, j),
                                                       desc_scale_atom(ssfa + 512 * j));
#pragma unroll
                        for (int h = 0; h < Cfg::kSfRb; ++h)
                            ptx::tc_cp_32x128b_warpx4_pair(
                                tmem_base + Cfg::sfb_col(stage, j, h),
                                desc_scale_atom(ssfb + Cfg::kMmas * 512 * h + 512 * j));
                    }
                    ptx::tc_commit_pair(sfr_bar(stage));
                    issued_any = true;
                }
            }
            if (issued_any) {
                ptx::tc_commit_pair(sf_drain_bar);
                wait_drain(sf_drain_bar, 0u, wctx);
            }
        }
    } else if (warp == Cfg::kMmaWarpP) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------ MMA issuer
            uint32_t q = 0;
            uint32_t acc_phase = 0;
            bool ok = true, issued_any = false;
            int g = 0;
            for (int t = pair; t < total && ok; t += npairs) {
                const TileCoord tc = tile_coord(p, t, g);
                const int nst = p.kchunks[tc.g];
                // both CTAs' epilogues have taken the previous tile out
                if (!wait_bounded(acce_bar, acc_phase ^ 1u, wctx, kRoleMma)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                for (int it = 0; it < nst; ++it, ++q) {
                    const int stage = (int)(q % S);
                    if (!wait_bounded(full_bar(stage), (q / S) & 1u, wctx, kRoleMma) ||
                        !wait_bounded(sfr_bar(stage), (q / S) & 1u, wctx, kRoleMma)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = base + stage * Cfg::kStageBytes;
                    const uint32_t sb = sa + Cfg::kABytes;
#pragma unroll
                    for (int j = 0; j < Cfg::kMmas; ++j)
                        ptx::tc_mma_nvfp4_pair(tmem_base, desc_operand_sw128(sa + 32 * j),
                                               desc_operand_sw128(sb + 32 * j), Cfg::kIdesc,
                                               tmem_base + Cfg::sfa_col(stage, j),
                                               tmem_base + Cfg::sfb_col(stage, j, 0),
                                               (it > 0 || j > 0) ? 1u : 0u);
                    // frees the slot in both CTAs
                    ptx::tc_commit_pair_mc(empty_bar(stage), (uint16_t)0x3);
                    issued_any = true;
                }
                if (!ok)
                    break;
                ptx::tc_commit_pair_mc(accf_bar, (uint16_t)0x3);
                acc_phase ^= 1u;
            }
            if (issued_any) {
                ptx::tc_commit_pair(drain_bar);
                wait_drain(drain_bar, 0u, wctx);
            }
        }
    } else if (warp < 4) {
        // ---------------------------------------------------- epilogue
        uint32_t acc_phase = 0;
        int g = 0;
        const uint32_t stage_buf = base + Cfg::kEpiOff + warp * Cfg::kEpiBufBytes;
        const uint32_t lane_tmem = (uint32_t)(warp * 32) << 16;
        const uint32_t acce_leader = ptx::mapa_shared(acce_bar, 0);
        for (int t = pair; t < total; t += npairs) {
            const TileCoord tc = tile_coord(p, t, g);
            uint32_t ready = 1u;
            if (lane == 0)
                ready = wait_bounded(accf_bar, acc_phase, wctx, kRoleEpilogue) ? 1u : 0u;
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (!ready)
                break;
            ptx::tc_fence_after();
            const int M = p.M[tc.g];
            const int N = p.N[tc.g];
            const int m0 = tc.bm * Cfg::kPairBM + (int)rank * kBM + warp * 32;
            const int n0 = tc.bn * BN;
            uint32_t h[BN / 2];
            if (m0 < M)
                epilogue_load<BN, EPI_EX>(p, tc.g, tmem_base + lane_tmem, n0, N, h);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive_cluster_relaxed(acce_leader);   // publishes no memory
            const bool sw = EPI_EX && p.swiglu;
            const int on0 = sw ? n0 / 2 : n0;     // output columns
            const int oN = sw ? N / 2 : N;
            const int ocols = sw ? BN / 2 : BN;
            // the CTA's last tile: every MMA has completed and no load is
            // left, so the operand ring is free -- each chunk gets its own
            // staging buffer there and the stores go out back to back
            const bool last_tile = t + npairs >= total;
            const uint32_t ring_buf = base + (uint32_t)(warp * (BN / EC)) * Cfg::kEpiBufBytes;
            if (m0 < M && last_tile && p.c_wide[tc.g]) {
                store_slab_wide<BN>(&p.tmCw[tc.g], base + (uint32_t)(warp * (BN / 64)) * 4096u, lane, on0, oN,
                                    ocols, m0, h);
            } else if (m0 < M) {
#pragma unroll
                for (int c = 0; c < BN / EC; ++c) {
                    if (c * EC < ocols && on0 + c * EC < oN) {   // warp-uniform
                        if (lane == 0 && !last_tile)
                            ptx::bulk_wait_group_read<0>();
                        __syncwarp();
                        const uint32_t buf = last_tile ? ring_buf + c * Cfg::kEpiBufBytes : stage_buf;
                        constexpr int kQ = EC / 8;
                        const uint32_t row = buf + lane * (EC * 2);
                        const int phase_r = (EC == 64) ? (lane & 7) : ((lane >> 1) & 3);
#pragma unroll
                        for (int q = 0; q < kQ; ++q)
                            ptx::st_shared_v4(row + ((q ^ phase_r) << 4), h[c * (EC / 2) + 4 * q],
                                              h[c * (EC / 2) + 4 * q + 1], h[c * (EC / 2) + 4 * q + 2],
                                              h[c * (EC / 2) + 4 * q + 3]);
                        ptx::fence_proxy_async_shared();
                        __syncwarp();
                        if (lane == 0) {
                            ptx::tma_store_2d(&p.tmC[tc.g], buf, on0 + c * EC, m0);
                            ptx::bulk_commit_group();
                        }
                        __syncwarp();
                    }
                }
            }
            acc_phase ^= 1u;
        }
        if (lane == 0)
            ptx::bulk_wait_group<0>();
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    // neither CTA leaves while the other may still signal it or read its
    // shared memory
    ptx::cluster_sync();
    if (warp == Cfg::kMmaWarpP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
    }
}

// 256 x 256 pair tiles, 5-stage ring (38 KiB per stage and CTA), 32-column
// epilogue stores
using CfgPair = PairConfig<256, 5, 32>;

}  // namespace nvfp4
