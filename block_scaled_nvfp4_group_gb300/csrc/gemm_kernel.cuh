// gemm_kernel.cuh -- persistent, warp-specialised NVFP4 grouped GEMM for
// sm_103a (GB300).
//
// One CTA per SM walks a flat list of output tiles of every group
// (tile t, t + gridDim.x, ...).  Six warps, three roles:
//   warps 0-3  epilogue: tensor memory -> registers (tcgen05.ld), FP32 ->
//              FP16 (round to nearest even), a swizzled shared-memory tile
//              per warp and a TMA tensor store, which writes whole 128-byte
//              row segments and clips rows >= M and columns >= N;
//   warp 4     producer: per 256-K stage, TMA loads of the A tile
//              [128 x 256] and the B tile [BN x 256] (128-byte swizzle) and
//              bulk copies of the matching tiled scale atoms into a ring of
//              STAGES shared-memory slots (mbarrier full/empty pairs);
//   warp 5     MMA issuer (one thread): tcgen05.cp of the stage's scale
//              atoms into tensor memory, four
//              tcgen05.mma.kind::mxf4nvf4.block_scale.block16 (128 x BN x 64)
//              per stage into a double-buffered FP32 accumulator, and
//              tcgen05.commit to free the stage / hand the accumulator on.
// The epilogue of tile t overlaps the MMAs of tile t+1.
//
// The warp split, the scale addressing and the descriptor fields follow
// kernelbot nvfp4-group-gemm submission 474067 (group_gemm_persistent_kernel,
// tcgen05_mma_nvfp4, tcgen05_cp_nvfp4, the TMA producer warp); the store
// path, the bounded waits and the tensor-memory budget are this build's own.
//
// Every mbarrier wait is bounded: when it expires the waiting role sets the
// device error word and a shared abort flag, all roles leave their loops, the
// producer waits (bounded) for the copies it issued, the MMA thread waits for
// its issued tensor-core work, the epilogue waits for its stores, and the CTA
// frees its tensor memory and exits.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"

namespace nvfp4 {

constexpr int kBM = 128;           // MMA M, rows of A per tile
constexpr int kBK = 256;           // K elements per pipeline stage
constexpr int kMmaK = 64;          // K elements per tcgen05.mma (FP4)
constexpr int kMaxGroups = 32;     // groups per launch (param block)
constexpr int kThreads = 192;      // 4 epilogue warps + producer + MMA
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kEpiBufBytes = 32 * 128;  // one warp's 32 rows x 64 FP16 columns

// error word bits (device_err[0]); device_err[1] records who expired first
constexpr uint32_t kErrTimeout = 1u;
constexpr uint32_t kErrDrainTimeout = 2u;

enum : uint32_t { kRoleProducer = 1, kRoleMma = 2, kRoleEpilogue = 3, kRoleDrain = 4 };

struct GemmParams {
    CUtensorMap tmA[kMaxGroups];  // uint8 [M][K/2], box 128 x 128 B, 128B swizzle
    CUtensorMap tmB[kMaxGroups];  // uint8 [N][K/2], box 128 x BN
    CUtensorMap tmC[kMaxGroups];  // fp16 [M][N], box 64 x 32, 128B swizzle
    const uint8_t *sfa[kMaxGroups];
    const uint8_t *sfb[kMaxGroups];
    int M[kMaxGroups];
    int N[kMaxGroups];
    int kiters[kMaxGroups];    // K / 256
    int grid_m[kMaxGroups];    // ceil(M / 128)
    int tile_end[kMaxGroups];  // inclusive prefix sum of grid_m * grid_n
    int num_groups;
    int total_tiles;
    uint32_t *err;             // device error words [2]
    unsigned long long timeout_ns;
    int b_policy;              // L2 policy of B / SFB loads: 0 normal, 1 first, 2 last
    int debug_drop_stage;      // test hook: CTA 0 never issues its first stage
};

template <int BN>
struct GemmConfig {
    static_assert(BN == 128 || BN == 256, "BN must be 128 or 256");
    static constexpr int kAccBufs = (BN == 128) ? 2 : 1;
    static constexpr int kStages = (BN == 128) ? 5 : 4;
    static constexpr int kABytes = kBM * kBK / 2;        // 16 KiB
    static constexpr int kBBytes = BN * kBK / 2;
    static constexpr int kSfaBytes = 4 * 512;            // 4 atoms (4 x 64 K)
    static constexpr int kSfbBytes = (BN / 128) * 4 * 512;
    static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1 KiB alignment");
    static constexpr int kEpiOff = kStages * kStageBytes;
    static constexpr int kBarOff = kEpiOff + 4 * 2 * kEpiBufBytes;
    // full[S], empty[S], acc_full[2], acc_empty[2], drain
    static constexpr int kNumBars = 2 * kStages + 5;
    static constexpr int kSlotOff = kBarOff + 8 * kNumBars;  // tmem base, abort flag
    static constexpr int kSmemBytes = kSlotOff + 16 + 1024;  // + alignment slack
    static_assert(kSmemBytes <= 232448, "exceeds 227 KiB of shared memory");
    // tensor memory: accumulators, then the scale columns of one stage
    static constexpr int kTmemCols = 512;
    static constexpr int kSfaCol = kAccBufs * BN;
    static constexpr int kSfbCol = kSfaCol + 4 * (kBK / kMmaK);
    static_assert(kSfbCol + 4 * (kBK / kMmaK) * (BN / 128) <= kTmemCols, "tensor memory budget");
    // instruction descriptor (kind::mxf4nvf4): A and B E2M1 (format 1) at
    // bits 7 and 10, both K-major, N>>3 at bit 17, UE4M3 scales (bit 23 = 0),
    // M>>7 at bit 27, scale-factor data ids 0
    static constexpr uint32_t kIdesc =
        (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kBM >> 7) << 27);
};

// shared-memory matrix descriptor, K-major operand tile with 128-byte
// swizzle: 8-row groups 1024 bytes apart, descriptor version 1 (bit 46)
__device__ __forceinline__ uint64_t desc_operand_sw128(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}

// descriptor of one 512-byte scale atom (32 rows x 16 bytes, no swizzle,
// 8-row groups 128 bytes apart)
__device__ __forceinline__ uint64_t desc_scale_atom(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 32) | (1ull << 46);
}

struct TileCoord {
    int g, bm, bn;
};

// advance the running group index to the group holding tile t (t only grows
// within one CTA) and split the group-local index, M-tile fastest, so that
// the M-tiles sharing one B strip are neighbours in the list
__device__ __forceinline__ TileCoord tile_coord(const GemmParams &p, int t, int &g)
{
    while (t >= p.tile_end[g])
        ++g;
    int local = t - (g > 0 ? p.tile_end[g - 1] : 0);
    int gm = p.grid_m[g];
    return TileCoord{g, local % gm, local / gm};
}

struct WaitCtx {
    volatile uint32_t *abort;
    uint32_t *err;
    unsigned long long timeout_ns;
};

__device__ __noinline__ bool wait_bounded_slow(uint32_t bar, uint32_t parity, const WaitCtx &w,
                                               uint32_t role)
{
    const uint64_t t0 = ptx::globaltimer_ns();
    for (;;) {
        if (ptx::mbar_try_wait(bar, parity))
            return true;
        if (*w.abort)
            return false;
        if (ptx::globaltimer_ns() - t0 > w.timeout_ns) {
            *w.abort = 1u;
            atomicOr(w.err, kErrTimeout);
            atomicCAS(w.err + 1, 0u, (blockIdx.x << 4) | role);
            return false;
        }
    }
}

// bounded wait: true once the phase completed; false when another role
// aborted or when this wait expired (then the error word and abort flag are
// set)
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtx &w,
                                             uint32_t role)
{
    if (ptx::mbar_try_wait(bar, parity))
        return true;
    return wait_bounded_slow(bar, parity, w, role);
}

// bounded wait used while draining after an abort (ignores the abort flag)
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity, const WaitCtx &w)
{
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > w.timeout_ns) {
            atomicOr(w.err, kErrDrainTimeout);
            atomicCAS(w.err + 1, 0u, (blockIdx.x << 4) | kRoleDrain);
            return;
        }
    }
}

__device__ __forceinline__ uint32_t pack_half2_rn(uint32_t lo_bits, uint32_t hi_bits)
{
    __half2 h = __floats2half2_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<uint32_t *>(&h);
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    nvfp4_group_gemm_kernel(const __grid_constant__ GemmParams p)
{
    using Cfg = GemmConfig<BN>;
    constexpr int S = Cfg::kStages;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);

    const uint32_t bar0 = base + Cfg::kBarOff;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * S + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * S + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
    const uint32_t tmem_slot = base + Cfg::kSlotOff;
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + Cfg::kSlotOff + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(accf_bar(b), 1);
            ptx::mbar_init(acce_bar(b), 4);  // lane 0 of each epilogue warp
        }
        ptx::mbar_init(drain_bar, 1);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == kProducerWarp) {
        ptx::tmem_alloc(tmem_slot, Cfg::kTmemCols);
        ptx::tmem_relinquish();
        ptx::tc_fence_before();
    }
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = ptx::ld_shared_u32(tmem_slot);

    const WaitCtx wctx{abort_flag, p.err, p.timeout_ns};
    const int total = p.total_tiles;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const uint64_t pol_a = ptx::policy_evict_last();
            const uint64_t pol_b = p.b_policy == 1   ? ptx::policy_evict_first()
                                   : p.b_policy == 2 ? ptx::policy_evict_last()
                                                     : ptx::policy_evict_normal();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issued_parity = 0;
            bool ok = true;
            int g = 0;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const TileCoord tc = tile_coord(p, t, g);
                const int kit = p.kiters[tc.g];
                const int kblk = kit * 4;  // 64-element K blocks per row block
                const CUtensorMap *tma = &p.tmA[tc.g];
                const CUtensorMap *tmb = &p.tmB[tc.g];
                const uint8_t *sfa = p.sfa[tc.g] + (size_t)tc.bm * kblk * 512;
                const uint8_t *sfb = p.sfb[tc.g] + (size_t)tc.bn * (BN / 128) * kblk * 512;
                for (int it = 0; it < kit; ++it) {
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, wctx, kRoleProducer)) {
                        ok = false;
                        break;
                    }
                    const bool drop = p.debug_drop_stage && blockIdx.x == 0 && t == (int)blockIdx.x &&
                                      it == 0;
                    if (!drop) {
                        const uint32_t sa = base + stage * Cfg::kStageBytes;
                        const uint32_t sb = sa + Cfg::kABytes;
                        const uint32_t ssfa = sb + Cfg::kBBytes;
                        const uint32_t ssfb = ssfa + Cfg::kSfaBytes;
                        const uint32_t fb = full_bar(stage);
                        ptx::mbar_arrive_expect_tx(fb, Cfg::kStageBytes);
                        ptx::tma_load_2d(sa, tma, it * (kBK / 2), tc.bm * kBM, fb, pol_a);
                        ptx::tma_load_2d(sb, tmb, it * (kBK / 2), tc.bn * BN, fb, pol_b);
                        ptx::bulk_load(ssfa, sfa + (size_t)it * 4 * 512, Cfg::kSfaBytes, fb, pol_a);
#pragma unroll
                        for (int h = 0; h < BN / 128; ++h)
                            ptx::bulk_load(ssfb + h * 2048, sfb + ((size_t)h * kblk + it * 4) * 512,
                                           2048, fb, pol_b);
                        issued |= 1u << stage;
                        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // copies issued but never consumed (after an abort anywhere in
            // the CTA) still land in this CTA's shared memory: wait for the
            // last issue of every slot before the CTA can exit (immediate on
            // the normal path, where the MMA thread consumed them all)
            (void)ok;
            for (int s = 0; s < S; ++s)
                if (issued & (1u << s))
                    wait_drain(full_bar(s), (issued_parity >> s) & 1u, wctx);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true, issued_any = false;
            int g = 0;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const TileCoord tc = tile_coord(p, t, g);
                const int kit = p.kiters[tc.g];
                if (!wait_bounded(acce_bar(acc), acc_phase ^ 1u, wctx, kRoleMma)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int it = 0; it < kit; ++it) {
                    if (!wait_bounded(full_bar(stage), phase, wctx, kRoleMma)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = base + stage * Cfg::kStageBytes;
                    const uint32_t sb = sa + Cfg::kABytes;
                    const uint32_t ssfa = sb + Cfg::kBBytes;
                    const uint32_t ssfb = ssfa + Cfg::kSfaBytes;
#pragma unroll
                    for (int j = 0; j < kBK / kMmaK; ++j) {
                        ptx::tc_cp_32x128b_warpx4(tmem_base + Cfg::kSfaCol + 4 * j,
                                                  desc_scale_atom(ssfa + 512 * j));
#pragma unroll
                        for (int h = 0; h < BN / 128; ++h)
                            ptx::tc_cp_32x128b_warpx4(
                                tmem_base + Cfg::kSfbCol + 4 * (BN / 128) * j + 4 * h,
                                desc_scale_atom(ssfb + 2048 * h + 512 * j));
                    }
#pragma unroll
                    for (int j = 0; j < kBK / kMmaK; ++j) {
                        ptx::tc_mma_nvfp4(d_tmem, desc_operand_sw128(sa + 32 * j),
                                          desc_operand_sw128(sb + 32 * j), Cfg::kIdesc,
                                          tmem_base + Cfg::kSfaCol + 4 * j,
                                          tmem_base + Cfg::kSfbCol + 4 * (BN / 128) * j,
                                          (it > 0 || j > 0) ? 1u : 0u);
                    }
                    ptx::tc_commit(empty_bar(stage));
                    issued_any = true;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                ptx::tc_commit(accf_bar(acc));
                if (++acc == Cfg::kAccBufs) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (issued_any) {
                // tensor-core work in flight still reads shared memory and
                // writes tensor memory: wait for all of it before teardown
                ptx::tc_commit(drain_bar);
                wait_drain(drain_bar, 0u, wctx);
            }
        }
    } else {
        // ---------------------------------------------------- epilogue
        int acc = 0;
        uint32_t acc_phase = 0;
        int sbuf = 0;
        int g = 0;
        const uint32_t stage_buf = base + Cfg::kEpiOff + warp * 2 * kEpiBufBytes;
        const uint32_t lane_tmem = (uint32_t)(warp * 32) << 16;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const TileCoord tc = tile_coord(p, t, g);
            // lane 0 waits; the outcome is broadcast so the warp stays
            // converged for the .sync.aligned tensor-memory loads
            uint32_t ready = 1u;
            if (lane == 0)
                ready = wait_bounded(accf_bar(acc), acc_phase, wctx, kRoleEpilogue) ? 1u : 0u;
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (!ready)
                break;
            ptx::tc_fence_after();
            const int M = p.M[tc.g];
            const int N = p.N[tc.g];
            const int m0 = tc.bm * kBM + warp * 32;
            const int n0 = tc.bn * BN;
            if (m0 < M) {
#pragma unroll 1
                for (int c = 0; c < BN / 64; ++c) {
                    if (n0 + c * 64 >= N)
                        break;
                    uint32_t v0[32], v1[32];
                    const uint32_t ta = tmem_base + lane_tmem + acc * BN + c * 64;
                    ptx::tmem_ld_32x32b_x32(ta, v0);
                    ptx::tmem_ld_32x32b_x32(ta + 32, v1);
                    ptx::tmem_wait_ld();
                    uint32_t h[32];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        h[i] = pack_half2_rn(v0[2 * i], v0[2 * i + 1]);
                        h[16 + i] = pack_half2_rn(v1[2 * i], v1[2 * i + 1]);
                    }
                    // the store that used this buffer two chunks ago must
                    // have finished reading it
                    if (lane == 0)
                        ptx::bulk_wait_group_read<1>();
                    __syncwarp();
                    const uint32_t buf = stage_buf + sbuf * kEpiBufBytes;
                    const uint32_t row = buf + lane * 128;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        ptx::st_shared_v4(row + ((q ^ (lane & 7)) << 4), h[4 * q], h[4 * q + 1],
                                          h[4 * q + 2], h[4 * q + 3]);
                    ptx::fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_2d(&p.tmC[tc.g], buf, n0 + c * 64, m0);
                        ptx::bulk_commit_group();
                    }
                    __syncwarp();
                    sbuf ^= 1;
                }
            }
            // every lane's loads have completed (wait::ld): hand the
            // accumulator back to the MMA thread
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(acce_bar(acc));
            if (++acc == Cfg::kAccBufs) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0)
            ptx::bulk_wait_group<0>();
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kProducerWarp) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
}

}  // namespace nvfp4
