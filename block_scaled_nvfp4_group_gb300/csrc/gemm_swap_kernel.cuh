// gemm_swap_kernel.cuh -- the NVFP4 grouped GEMM for small M (MoE-shaped
// calls) on CTA pairs, with the operands' roles swapped (sm_103a).
//
// C_g = A_g . B_g^T is computed as its transpose C_g^T = B_g . A_g^T: the
// rows of B_g (the N side, e.g. an expert's weights) are the MMA's M = 256
// side, split 128 / 128 over the two CTAs of a cluster, and the rows of A_g
// (the M_g tokens of the group, at most 256 per tile) are the MMA's N side,
// N = M_g rounded up to 16, half of them staged by each CTA.  So
//   * a tile is (group, 256 rows of B, one token tile of <= 256 rows of A):
//     every byte of B leaves L2 once per token tile (groups of <= 256 rows:
//     once), where 128-row M tiles would stream it once per M tile;
//   * the MMA does no work on padding rows past M_g beyond the rounding to 16
//     (128-row M tiles pad M_g = 45 to 128);
//   * the accumulator holds D[n][m]: tensor-memory lane = row of B (column of
//     C), column = token (row of C), so the epilogue transposes through shared
//     memory before its TMA stores.
// Groups with more than 256 rows are split by the host into token tiles of
// at most 256 rows (a multiple of 128 rows apart, where the tiled scales of
// A start a new 128-row block), each its own entry with offset pointers.
//
// Roles (warps, both CTAs unless noted) as in gemm_pair_kernel.cuh:
//   0-3  epilogue: this CTA's 128 rows of B (accumulator lanes) x the tile's
//        tokens -> FP16 (or BF16 x alpha) -> 32 x 32 blocks transposed into
//        shared memory -> TMA tensor stores of C;
//   4    MMA issuer (even CTA, one thread);
//   5    scale copier (even CTA, one thread);
//   6-9  loaders: this CTA's 128 rows of B, its half of the tile's token rows
//        (on full[slot]), the scale atoms of its 128 B rows and those of all
//        the tile's token rows (on sf_full[slot]);
//   10   L2 prefetcher of this CTA's B rows.
//
// The tile roles, descriptors and the scale-atom addressing follow kernelbot
// nvfp4-group-gemm submission 474067 (group_gemm_persistent_kernel,
// tcgen05_mma_nvfp4, tcgen05_cp_nvfp4); the swapped operand roles, the token
// tiles, the CTA pairs, the transposing epilogue and the bounded waits are
// this build's own.
#pragma once

#include "gemm_pair_kernel.cuh"

namespace nvfp4 {

constexpr int kSwapMaxW = 16;      // groups (B matrices) per launch
constexpr int kSwapMaxT = 32;      // token tiles per launch
constexpr int kSwapMaxTok = 256;   // token rows per tile (the MMA's largest N)

struct SwapParams {
    CUtensorMap tmW[kSwapMaxW];    // B_g: uint8 {128 B, N, K/256}, box {128, 128, 1}
    CUtensorMap tmSW[kSwapMaxW];   // tiled SFB_g: uint32 {128, K/64, N blocks}, box {128, 4, 1}
    CUtensorMap tmX[kSwapMaxT];    // the tile's rows of A_g: uint8 {128 B, Mt, K/256}, box {128, npad/2, 1}
    CUtensorMap tmSX[kSwapMaxT];   // their tiled SFA: {128, K/64, ceil(Mt/128)}, box {128, 4, ceil(Mt/128)}
    CUtensorMap tmC[kSwapMaxT];    // the tile's rows of C: 16-bit {N, Mt}, box {32, 32}, no swizzle
    int t_group[kSwapMaxT];        // group (index into the w_ arrays) of token tile t
    int t_rows[kSwapMaxT];         // Mt, 1..256
    int t_npad[kSwapMaxT];         // MMA N: Mt rounded up to 16
    int t_sfx[kSwapMaxT];          // 128-row scale blocks of the tile's tokens (1 or 2)
    int w_N[kSwapMaxW];
    int w_kchunks[kSwapMaxW];      // K / 256 (= stages of a tile)
    int w_tiles[kSwapMaxW];        // ceil(N / 256): tiles of 256 rows of B
    int w_tfirst[kSwapMaxW];       // token tiles of group g: [w_tfirst, w_tfirst + w_tcount)
    int w_tcount[kSwapMaxW];
    int tile_end[kSwapMaxW];       // inclusive prefix sum of w_tiles * w_tcount
    float alpha[kSwapMaxW];
    int num_w;
    int total_tiles;
    int out_bf16;                  // C elements: 0 FP16, 1 BF16
    int early_ab;                  // A and B complete before the preceding kernel began
    int b_policy;
    int pf_stages;
    int debug_drop_stage;
    uint32_t *err;
    unsigned long long timeout_ns;
};
static_assert(sizeof(SwapParams) <= 32764, "kernel parameter block over 32 KiB");

template <int STAGES_>
struct SwapConfig {
    static constexpr int kStages = STAGES_;
    static constexpr int BW = 256;                          // rows of B per tile (MMA M)
    static constexpr int kMmas = kChunkK / kMmaK;           // 4 per 256-K stage
    static constexpr int kWBytes = kBM * 128;               // this CTA's 128 rows of B, 16 KiB
    static constexpr int kXBytes = (kSwapMaxTok / 2) * 128; // up to 128 token rows, 16 KiB
    static constexpr int kSwBytes = kMmas * 512;            // one 128-row block of B scales
    static constexpr int kSxBytes = 2 * kMmas * 512;        // up to two blocks of token scales
    static constexpr int kStageBytes = kWBytes + kXBytes + kSwBytes + kSxBytes;
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1 KiB alignment");
    static constexpr int kEpiBufBytes = 32 * 32 * 2;        // 32 tokens x 32 columns of C
    static constexpr int kEpiOff = kStages * kStageBytes;
    static constexpr int kBarOff = kEpiOff + 4 * 2 * kEpiBufBytes;
    // full[S], empty[S], sf_ready[S], sf_full[S], acc_full, acc_empty, drain, sf_drain
    static constexpr int kNumBars = 4 * kStages + 4;
    static constexpr int kSlotOff = kBarOff + 8 * kNumBars;
    static constexpr int kSmemBytes = kSlotOff + 16 + 1024;
    static_assert(kSmemBytes <= kSmemLimit, "exceeds 227 KiB of shared memory");
    static constexpr int kMmaWarp = 4;
    static constexpr int kSfWarp = 5;
    static constexpr int kFirstLoader = 6;   // B rows, token rows, B scales, token scales
    static constexpr int kPrefetchWarp = 10;
    static constexpr int kThreads = 32 * (kPrefetchWarp + 1);
    static constexpr int kTmemCols = 512;
    static constexpr int kSfCol0 = kSwapMaxTok;             // one accumulator of up to 256 columns
    static constexpr int kSfSlotCols = 4 * kMmas * 3;       // per k block: 1 B atom, 2 token atoms
    static_assert(kSfCol0 + kStages * kSfSlotCols <= kTmemCols, "tensor memory budget");
    static constexpr uint32_t sfw_col(int slot, int j) { return kSfCol0 + slot * kSfSlotCols + 4 * j; }
    static constexpr uint32_t sfx_col(int slot, int j, int h)
    {
        return kSfCol0 + slot * kSfSlotCols + 4 * kMmas + 8 * j + 4 * h;
    }
    // kind::mxf4nvf4 instruction descriptor: E2M1 A and B, K-major, UE4M3
    // scales, M = 256 (CTA pair), N = npad (a multiple of 16, 16..256)
    static __device__ __forceinline__ uint32_t idesc(int npad)
    {
        return (1u << 7) | (1u << 10) | ((uint32_t)(npad >> 3) << 17) | ((uint32_t)(BW >> 7) << 27);
    }
};

struct SwapTile {
    int g;    // group
    int nb;   // tile of 256 rows of B
    int t;    // token tile
};

// tile list: for every group, for every 256-row tile of B, its token tiles
// in order (token tile fastest, so the tiles sharing a B tile run on
// neighbouring pairs at the same time and share its bytes through L2);
// `g` is a running group index (tiles only grow within one pair)
__device__ __forceinline__ SwapTile swap_tile(const SwapParams &p, int tile, int &g)
{
    while (tile >= p.tile_end[g])
        ++g;
    const int local = tile - (g > 0 ? p.tile_end[g - 1] : 0);
    const int tc = p.w_tcount[g];
    return SwapTile{g, local / tc, p.w_tfirst[g] + local % tc};
}

// One loader of one CTA of the pair: ROLE 0 this CTA's 128 rows of B, 1 its
// half of the tile's token rows (both on full[slot]), 2 the scale atoms of
// its 128 rows of B, 3 the scale atoms of all the tile's token rows (both on
// sf_full[slot]).  Loads complete on the even CTA's barrier; only the even
// CTA's loaders arrive there, with the bytes of both CTAs.  Boxes reaching
// past N, Mt or K land as zeros and count their full size.
template <class Cfg, int ROLE>
__device__ __forceinline__ void swap_loader(const SwapParams &p, uint32_t base, uint32_t bar0, uint32_t rank,
                                            volatile uint32_t *w_progress, const WaitCtx &wctx)
{
    constexpr int S = Cfg::kStages;
    constexpr bool kSf = ROLE >= 2;
    constexpr uint32_t kOff = ROLE == 0   ? 0u
                              : ROLE == 1 ? (uint32_t)Cfg::kWBytes
                              : ROLE == 2 ? (uint32_t)(Cfg::kWBytes + Cfg::kXBytes)
                                          : (uint32_t)(Cfg::kWBytes + Cfg::kXBytes + Cfg::kSwBytes);
    auto done_bar = [&](int s) { return bar0 + 8u * ((kSf ? 3 * S : 0) + s); };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };

    const bool w_side = (ROLE == 0 || ROLE == 2);
    const uint64_t pol = w_side ? (p.b_policy == 1   ? ptx::policy_evict_first()
                                   : p.b_policy == 2 ? ptx::policy_evict_last()
                                                     : ptx::policy_evict_normal())
                                : ptx::policy_evict_last();
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
    uint32_t q = 0;
    uint32_t issued = 0, issued_parity = 0;
    bool ok = true;
    int g = 0;
    for (int tile = pair; tile < p.total_tiles && ok; tile += npairs) {
        const SwapTile tc = swap_tile(p, tile, g);
        const int nst = p.w_kchunks[tc.g];
        const int xrows = p.t_npad[tc.t] / 2;
        const uint32_t tx = ROLE == 0   ? 2u * Cfg::kWBytes
                            : ROLE == 1 ? 2u * (uint32_t)xrows * 128u
                            : ROLE == 2 ? 2u * Cfg::kSwBytes
                                        : 2u * (uint32_t)p.t_sfx[tc.t] * (uint32_t)(Cfg::kMmas * 512);
        for (int it = 0; it < nst; ++it, ++q) {
            const int stage = (int)(q % S);
            const uint32_t phase = (q / S) & 1u;
            if (!wait_bounded(empty_bar(stage), phase ^ 1u, wctx, kRoleProducer)) {
                ok = false;
                break;
            }
            const bool drop = ROLE == 0 && p.debug_drop_stage && blockIdx.x == 0 && q == 0;
            if (!drop) {
                const uint32_t dst = base + stage * Cfg::kStageBytes + kOff;
                const uint32_t bar_leader = ptx::mapa_shared(done_bar(stage), 0);
                if (rank == 0)
                    ptx::mbar_arrive_expect_tx(done_bar(stage), tx);
                if (ROLE == 0)
                    ptx::tma_load_3d_pair(dst, &p.tmW[tc.g], 0, tc.nb * Cfg::BW + (int)rank * kBM, it, bar_leader,
                                          pol);
                else if (ROLE == 1)
                    ptx::tma_load_3d_pair(dst, &p.tmX[tc.t], 0, (int)rank * xrows, it, bar_leader, pol);
                else if (ROLE == 2)
                    ptx::tma_load_3d_pair(dst, &p.tmSW[tc.g], 0, it * Cfg::kMmas, tc.nb * 2 + (int)rank,
                                          bar_leader, pol);
                else
                    ptx::tma_load_3d_pair(dst, &p.tmSX[tc.t], 0, it * Cfg::kMmas, 0, bar_leader, pol);
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            }
            if (ROLE == 0)
                *w_progress = q + 1;
        }
    }
    (void)ok;
    // loads issued but not consumed still land in this CTA's shared memory:
    // the even CTA waits for its own barriers' phases (they count both CTAs'
    // bytes); the odd CTA waits for the MMAs to release its slots, giving up
    // at the first expiry
    bool alive = true;
    for (int s = 0; s < S && alive; ++s) {
        if (!(issued & (1u << s)))
            continue;
        const uint32_t par = (issued_parity >> s) & 1u;
        alive = rank == 0 ? wait_drain_ok(done_bar(s), par, wctx) : wait_drain_ok(empty_bar(s), par, wctx);
    }
}

// L2 prefetch of this CTA's 128 rows of B and their scale block, up to
// `pf_stages` stages ahead of this CTA's B loader; a B tile shared by
// consecutive token tiles is prefetched for its first token tile only
template <class Cfg>
__device__ __forceinline__ void swap_prefetch(const SwapParams &p, uint32_t rank, volatile uint32_t *w_progress,
                                              const WaitCtx &wctx)
{
    const uint64_t pol = p.b_policy == 1   ? ptx::policy_evict_first()
                         : p.b_policy == 2 ? ptx::policy_evict_last()
                                           : ptx::policy_evict_normal();
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
    uint32_t q = 0;
    int g = 0;
    for (int tile = pair; tile < p.total_tiles; tile += npairs) {
        const SwapTile tc = swap_tile(p, tile, g);
        const int nst = p.w_kchunks[tc.g];
        const bool first = tc.t == p.w_tfirst[tc.g];
        const int row0 = tc.nb * Cfg::BW + (int)rank * kBM;
        for (int it = 0; it < nst; ++it, ++q) {
            if (!first)
                continue;
            if (q >= *w_progress + (uint32_t)p.pf_stages) {
                const uint64_t t0 = ptx::globaltimer_ns();
                while (q >= *w_progress + (uint32_t)p.pf_stages) {
                    if (*wctx.abort || ptx::globaltimer_ns() - t0 > wctx.timeout_ns)
                        return;
                    __nanosleep(128);
                }
            }
            ptx::tma_prefetch_3d(&p.tmW[tc.g], 0, row0, it, pol);
            ptx::tma_prefetch_3d(&p.tmSW[tc.g], 0, it * Cfg::kMmas, tc.nb * 2 + (int)rank, pol);
        }
    }
}

template <class Cfg, bool EPI_EX>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    nvfp4_group_gemm_swap_kernel(const __grid_constant__ SwapParams p)
{
    constexpr int S = Cfg::kStages;

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
    volatile uint32_t *w_progress = reinterpret_cast<volatile uint32_t *>(gbase + Cfg::kSlotOff + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full_bar(s), 2);     // the even CTA's B-row and token-row loaders
            ptx::mbar_init(empty_bar(s), 1);
            ptx::mbar_init(sfr_bar(s), 1);
            ptx::mbar_init(sffull_bar(s), 2);   // the even CTA's scale loaders
        }
        ptx::mbar_init(accf_bar, 1);
        ptx::mbar_init(acce_bar, 8);          // lane 0 of the 4 epilogue warps of both CTAs
        ptx::mbar_init(drain_bar, 1);
        ptx::mbar_init(sf_drain_bar, 1);
        *abort_flag = 0u;
        *w_progress = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == Cfg::kMmaWarp) {
        ptx::tmem_alloc_pair(tmem_slot, Cfg::kTmemCols);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();   // both CTAs' barriers exist before either signals the other
    ptx::tc_fence_after();
    const uint32_t tmem_base = ptx::ld_shared_u32(tmem_slot);
    if (!(p.early_ab && (warp == Cfg::kFirstLoader || warp == Cfg::kFirstLoader + 1)))
        ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();

    const WaitCtx wctx{abort_flag, p.err, p.timeout_ns};
    const int total = p.total_tiles;
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);

    if (warp == Cfg::kPrefetchWarp) {
        if (lane == 0 && p.pf_stages > 0)
            swap_prefetch<Cfg>(p, rank, w_progress, wctx);
    } else if (warp >= Cfg::kFirstLoader) {
        if (lane == 0) {
            switch (warp - Cfg::kFirstLoader) {
            case 0: swap_loader<Cfg, 0>(p, base, bar0, rank, w_progress, wctx); break;
            case 1: swap_loader<Cfg, 1>(p, base, bar0, rank, w_progress, wctx); break;
            case 2: swap_loader<Cfg, 2>(p, base, bar0, rank, w_progress, wctx); break;
            default: swap_loader<Cfg, 3>(p, base, bar0, rank, w_progress, wctx); break;
            }
        }
    } else if (warp == Cfg::kSfWarp) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------- scale copies
            uint32_t q = 0;
            bool ok = true, issued_any = false;
            int g = 0;
            for (int tile = pair; tile < total && ok; tile += npairs) {
                const SwapTile tc = swap_tile(p, tile, g);
                const int nst = p.w_kchunks[tc.g];
                const int nsx = p.t_sfx[tc.t];
                for (int it = 0; it < nst; ++it, ++q) {
                    const int stage = (int)(q % S);
                    if (!wait_bounded(sffull_bar(stage), (q / S) & 1u, wctx, kRoleSf)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t ssw = base + stage * Cfg::kStageBytes + Cfg::kWBytes + Cfg::kXBytes;
                    const uint32_t ssx = ssw + Cfg::kSwBytes;
#pragma unroll
                    for (int j = 0; j < Cfg::kMmas; ++j) {
                        ptx::tc_cp_32x128b_warpx4_pair(tmem_base + Cfg::sfw_col(stage, j),
                                                       desc_scale_atom(ssw + 512 * j));
                        for (int h = 0; h < nsx; ++h)
                            ptx::tc_cp_32x128b_warpx4_pair(tmem_base + Cfg::sfx_col(stage, j, h),
                                                           desc_scale_atom(ssx + Cfg::kMmas * 512 * h + 512 * j));
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
    } else if (warp == Cfg::kMmaWarp) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------ MMA issuer
            uint32_t q = 0;
            uint32_t acc_phase = 0;
            bool ok = true, issued_any = false;
            int g = 0;
            for (int tile = pair; tile < total && ok; tile += npairs) {
                const SwapTile tc = swap_tile(p, tile, g);
                const int nst = p.w_kchunks[tc.g];
                const uint32_t idesc = Cfg::idesc(p.t_npad[tc.t]);
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
                    const uint32_t sw = base + stage * Cfg::kStageBytes;
                    const uint32_t sx = sw + Cfg::kWBytes;
#pragma unroll
                    for (int j = 0; j < Cfg::kMmas; ++j)
                        ptx::tc_mma_nvfp4_pair(tmem_base, desc_operand_sw128(sw + 32 * j),
                                               desc_operand_sw128(sx + 32 * j), idesc,
                                               tmem_base + Cfg::sfw_col(stage, j),
                                               tmem_base + Cfg::sfx_col(stage, j, 0), (it > 0 || j > 0) ? 1u : 0u);
                    ptx::tc_commit_pair_mc(empty_bar(stage), (uint16_t)0x3);   // frees the slot in both CTAs
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
        int sbuf = 0;
        const uint32_t stage_buf = base + Cfg::kEpiOff + warp * 2 * Cfg::kEpiBufBytes;
        uint16_t *const stage_ptr = reinterpret_cast<uint16_t *>(gbase + Cfg::kEpiOff + warp * 2 * Cfg::kEpiBufBytes);
        const uint32_t lane_tmem = (uint32_t)(warp * 32) << 16;
        const uint32_t acce_leader = ptx::mapa_shared(acce_bar, 0);
        for (int tile = pair; tile < total; tile += npairs) {
            const SwapTile tc = swap_tile(p, tile, g);
            uint32_t ready = 1u;
            if (lane == 0)
                ready = wait_bounded(accf_bar, acc_phase, wctx, kRoleEpilogue) ? 1u : 0u;
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (!ready)
                break;
            ptx::tc_fence_after();
            const int N = p.w_N[tc.g];
            const int Mt = p.t_rows[tc.t];
            const int nch = (Mt + 31) / 32;                       // 32-token chunks
            const int col0 = tc.nb * Cfg::BW + (int)rank * kBM + warp * 32;   // column of C of lane 0
            const bool live = col0 < N;                            // warp-uniform
            // 1. this thread's accumulator row (one column of C) -> 16-bit
            // pairs of neighbouring tokens in registers
            uint32_t h[kSwapMaxTok / 2];
            if (live) {
                const float alpha = EPI_EX ? p.alpha[tc.g] : 1.0f;
                const bool bf = EPI_EX && p.out_bf16 != 0;
#pragma unroll
                for (int c = 0; c < kSwapMaxTok / 32; ++c) {
                    if (c < nch) {   // warp-uniform
                        uint32_t v[32];
                        ptx::tmem_ld_32x32b_x32(tmem_base + lane_tmem + c * 32, v);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float lo = __uint_as_float(v[2 * i]), hi = __uint_as_float(v[2 * i + 1]);
                            if (EPI_EX) {
                                lo *= alpha;
                                hi *= alpha;
                            }
                            h[c * 16 + i] = pack_out2(lo, hi, bf);
                        }
                    }
                }
            }
            // 2. the accumulator goes back to the even CTA's MMA thread
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive_cluster_relaxed(acce_leader);   // publishes no memory
            // 3. 32 x 32 blocks (32 tokens x this warp's 32 columns of C),
            // transposed into shared memory (row = token, 64 bytes), each
            // stored with one TMA tensor store; two staging buffers per warp
            if (live) {
#pragma unroll
                for (int c = 0; c < kSwapMaxTok / 32; ++c) {
                    if (c < nch) {   // warp-uniform
                        if (lane == 0)
                            ptx::bulk_wait_group_read<1>();
                        __syncwarp();
                        uint16_t *const buf = stage_ptr + sbuf * (Cfg::kEpiBufBytes / 2);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            buf[(2 * i) * 32 + lane] = (uint16_t)(h[c * 16 + i] & 0xFFFFu);
                            buf[(2 * i + 1) * 32 + lane] = (uint16_t)(h[c * 16 + i] >> 16);
                        }
                        ptx::fence_proxy_async_shared();
                        __syncwarp();
                        if (lane == 0) {
                            ptx::tma_store_2d(&p.tmC[tc.t], stage_buf + sbuf * Cfg::kEpiBufBytes, col0, c * 32);
                            ptx::bulk_commit_group();
                        }
                        __syncwarp();
                        sbuf ^= 1;
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
    if (warp == Cfg::kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
    }
}

// 5-stage ring (38 KiB per stage and CTA)
using CfgSwap = SwapConfig<5>;

}  // namespace nvfp4
