// group_gemm.cu -- C-ABI entry points nvfp4_group_gemm and
// nvfp4_group_gemm_noalloc: validation, the per-call tile plan, the kernel
// configuration for the shape class, tensor maps and the launches of the
// persistent kernel.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/nvfp4_group_gemm.h"
#include "gemm_swap_kernel.cuh"
#include "runtime.h"

namespace nvfp4 {
namespace {

constexpr int kMaxDim = 1 << 20;
constexpr int kMaxGroupsPerCall = 4096;
constexpr long long kMaxTilesPerLaunch = 1ll << 30;
constexpr int kMaxDevices = 64;

// kernel configurations: the NVFP4_KIND_* numbers of the C ABI
enum Kind : int {
    kKindStream = NVFP4_KIND_STREAM,
    kKindWide = NVFP4_KIND_WIDE,
    kKindCompute = NVFP4_KIND_COMPUTE,
    kKindWide512 = NVFP4_KIND_WIDE512,
    kKindWideP2 = NVFP4_KIND_WIDE_P2,
    kKindWideP4 = NVFP4_KIND_WIDE_P4,
    kKindPair = NVFP4_KIND_PAIR,
    kKindWideSK = NVFP4_KIND_WIDE_SK,
    kKindSwap = NVFP4_KIND_SWAP,
    kNumKinds = 9
};

bool needs_n256(int kind)
{
    return kind == kKindWide || kind == kKindWide512 || kind == kKindWideP2 || kind == kKindWideP4 ||
           kind == kKindWideSK;
}

// the producer-pair variants are folded into WIDE: every stage's loads are
// spread over four issuing warps in every configuration
int canonical_kind(int kind)
{
    return (kind == kKindWideP2 || kind == kKindWideP4) ? kKindWide : kind;
}

// Launch configuration shared by every kind: programmatic stream
// serialization (unless NVFP4_PDL=0), so the kernel may start while the
// previous kernel in the stream finishes and waits for it
// (griddepcontrol.wait) before touching global memory; CTA pairs also get a
// cluster of two.
struct LaunchCfg {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
};

void make_launch_cfg(LaunchCfg &L, int grid, int threads, int smem, bool pair, cudaStream_t s)
{
    L.cfg = cudaLaunchConfig_t{};
    L.cfg.gridDim = dim3(grid);
    L.cfg.blockDim = dim3(threads);
    L.cfg.dynamicSmemBytes = smem;
    L.cfg.stream = s;
    L.attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    L.attr[0].val.programmaticStreamSerializationAllowed = env_int("NVFP4_PDL", 1) != 0;
    L.attr[1].id = cudaLaunchAttributeClusterDimension;
    L.attr[1].val.clusterDim.x = 2;
    L.attr[1].val.clusterDim.y = 1;
    L.attr[1].val.clusterDim.z = 1;
    L.cfg.attrs = L.attr;
    L.cfg.numAttrs = pair ? 2 : 1;
}

template <class Cfg, bool SK>
cudaError_t launch_kind(const KernelParams &P, int grid, cudaStream_t s, bool ex)
{
    LaunchCfg L;
    make_launch_cfg(L, grid, Cfg::kThreads, Cfg::kSmemBytes, false, s);
    return ex ? cudaLaunchKernelEx(&L.cfg, nvfp4_group_gemm_kernel<Cfg, true, SK>, P)
              : cudaLaunchKernelEx(&L.cfg, nvfp4_group_gemm_kernel<Cfg, false, SK>, P);
}

template <class Cfg>
cudaError_t launch_pair_kind(const KernelParams &P, int grid, cudaStream_t s, bool ex)
{
    LaunchCfg L;
    make_launch_cfg(L, grid, Cfg::kThreads, Cfg::kSmemBytes, true, s);
    return ex ? cudaLaunchKernelEx(&L.cfg, nvfp4_group_gemm_pair_kernel<Cfg, true>, P)
              : cudaLaunchKernelEx(&L.cfg, nvfp4_group_gemm_pair_kernel<Cfg, false>, P);
}

struct KindInfo {
    int bm;         // output rows per tile (256 for CTA pairs)
    int bn;
    int box_b;      // rows of B one CTA loads per stage
    int chunks;     // 128-byte K chunks per row per stage
    int sf_atoms;   // scale atoms per row block per stage (stage K / 64)
    int sfb_blocks; // 128-row scale blocks of B per stage
    int epi_cols;
    int threads;
    int smem;
    bool pair;
    bool sk;             // stream-K ranges of (tile, stage) units
    const void *fn;      // plain FP16 epilogue
    const void *fn_ex;   // fused epilogue options compiled in
    cudaError_t (*launch)(const KernelParams &, int, cudaStream_t, bool);
};

template <class Cfg, bool SK = false>
KindInfo make_kind()
{
    return KindInfo{kBM, Cfg::BN, Cfg::BN, Cfg::kChunks, Cfg::kMmas, Cfg::BN / 128, Cfg::kEpiCols,
                    Cfg::kThreads, Cfg::kSmemBytes, false, SK,
                    reinterpret_cast<const void *>(&nvfp4_group_gemm_kernel<Cfg, false, SK>),
                    reinterpret_cast<const void *>(&nvfp4_group_gemm_kernel<Cfg, true, SK>),
                    &launch_kind<Cfg, SK>};
}

template <class Cfg>
KindInfo make_pair_kind()
{
    return KindInfo{Cfg::kPairBM, Cfg::BN, Cfg::BN / 2, 1, Cfg::kMmas, Cfg::kSfRb, Cfg::kEpiCols,
                    Cfg::kThreads, Cfg::kSmemBytes, true, false,
                    reinterpret_cast<const void *>(&nvfp4_group_gemm_pair_kernel<Cfg, false>),
                    reinterpret_cast<const void *>(&nvfp4_group_gemm_pair_kernel<Cfg, true>),
                    &launch_pair_kind<Cfg>};
}

// the swapped-operand pair kernel takes its own parameter block
// (plan_and_launch_swap); its entry here serves the attributes and the
// cluster occupancy query only
KindInfo make_swap_kind()
{
    return KindInfo{CfgSwap::BW, kSwapMaxTok, kBM, 1, CfgSwap::kMmas, 1, 32, CfgSwap::kThreads,
                    CfgSwap::kSmemBytes, true, false,
                    reinterpret_cast<const void *>(&nvfp4_group_gemm_swap_kernel<CfgSwap, false>),
                    reinterpret_cast<const void *>(&nvfp4_group_gemm_swap_kernel<CfgSwap, true>), nullptr};
}

const KindInfo &kind_info(int k)
{
    static const KindInfo table[kNumKinds] = {
        make_kind<CfgStream>(),  make_kind<CfgWide>(), make_kind<CfgCompute>(),
        make_kind<CfgWide512>(), make_kind<CfgWide>(), make_kind<CfgWide>(),
        make_pair_kind<CfgPair>(), make_kind<CfgWide, true>(), make_swap_kind()};
    return table[canonical_kind(k)];
}

std::mutex g_attr_mu;
bool g_attr_set[kMaxDevices][kNumKinds];
int g_max_pairs[kMaxDevices][kNumKinds];

// Shared-memory attribute of the kind's kernel on this device and, for CTA
// pairs, how many pairs can be resident at once (the persistent grid size)
int ensure_kernel_attributes(int dev, int kind)
{
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (dev < 0 || dev >= kMaxDevices)
        return NVFP4_ERR_UNSUPPORTED;
    if (!g_attr_set[dev][kind]) {
        const KindInfo &ki = kind_info(kind);
        if (cudaFuncSetAttribute(ki.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ki.smem) !=
                cudaSuccess ||
            cudaFuncSetAttribute(ki.fn_ex, cudaFuncAttributeMaxDynamicSharedMemorySize, ki.smem) !=
                cudaSuccess)
            return NVFP4_ERR_CUDA;
        if (ki.pair) {
            LaunchCfg L;
            make_launch_cfg(L, 2, ki.threads, ki.smem, true, nullptr);
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, ki.fn, &L.cfg) != cudaSuccess ||
                clusters < 1)
                return NVFP4_ERR_UNSUPPORTED;
            g_max_pairs[dev][kind] = clusters;
        }
        g_attr_set[dev][kind] = true;
    }
    return NVFP4_OK;
}

// persistent grid of a launch with `tiles` tiles
int grid_size(int dev, int kind, int tiles, int sm_count)
{
    if (kind_info(kind).pair) {
        const int pairs = g_max_pairs[dev][kind];
        return 2 * (tiles < pairs ? tiles : pairs);
    }
    return tiles < sm_count ? tiles : sm_count;
}

int validate_group(const GroupDesc &g)
{
    if (g.M < 0 || g.N < 8 || g.K < 256 || g.M > kMaxDim || g.N > kMaxDim || g.K > kMaxDim)
        return NVFP4_ERR_INVALID_ARGUMENT;
    if (g.N % 8 != 0 || g.K % 256 != 0)
        return NVFP4_ERR_INVALID_ARGUMENT;
    if (g.M == 0)
        return NVFP4_OK;
    if (!g.A || !g.B || !g.SFA || !g.SFB || !g.C)
        return NVFP4_ERR_INVALID_ARGUMENT;
    if (!aligned16(g.A) || !aligned16(g.B) || !aligned16(g.SFA) || !aligned16(g.SFB) ||
        !aligned16(g.C))
        return NVFP4_ERR_MISALIGNED;
    return NVFP4_OK;
}

int validate_call(const GroupDesc *groups, int num_groups)
{
    if (!groups || num_groups < 1)
        return NVFP4_ERR_INVALID_ARGUMENT;
    if (num_groups > kMaxGroupsPerCall)
        return NVFP4_ERR_TOO_MANY;
    for (int i = 0; i < num_groups; ++i) {
        int rc = validate_group(groups[i]);
        if (rc != NVFP4_OK)
            return rc;
    }
    return NVFP4_OK;
}

// Kernel configuration of a call.  BN = 256 tiles (CfgWide) halve the A
// re-reads and the TMA operations per output byte, which the measurements on
// GB300 show matters for every shape here; they need every N to be a multiple
// of 256 (a B tile takes two whole 128-row scale blocks).  Otherwise BN = 128
// with 512-K stages (CfgStream).  A call that fits one round of the grid in
// 128 x 128 tiles runs them (CfgCompute).  CTA pairs (CfgPair, 256 x 256
// tiles) run a 256 x 256 tile in about 0.92 of the time one CTA takes for a
// 128 x 256 tile, but pad M to 256: they are chosen when pairing does not
// add a round of the grid (large M, e.g. the 4096^3 groups, and calls of
// fewer tiles than SMs), never for the small-M MoE shapes.  Stream-K (WIDE_SK) is
// never chosen here: on GB300 it measured slower than whole tiles even where
// it removes the most idle time (fewer tiles than SMs: 2 groups of 512 x
// 3072 x 4096, 33.7 vs 21.2 us): its ranges start at scattered K offsets, so
// the first loads pull far more distinct bytes from HBM, each stage then
// competes with 152 instead of 96 CTAs, and the cut tiles add a partial-sum
// exchange.  NVFP4_GEMM_KIND overrides the choice.
int choose_kind(const GroupDesc *groups, int n, int sm_count, bool need_bn256 = false)
{
    const int forced_env = env_int("NVFP4_GEMM_KIND", -1);
    // SwiGLU pairs the two 128-column halves of a 256-column tile
    const int forced = (need_bn256 && forced_env >= 0 && forced_env < kNumKinds &&
                        (kind_info(forced_env).bn != 256 || forced_env == kKindSwap))
                           ? kKindWide
                           : forced_env;
    bool all_n256 = true, all_n_ge256 = true;
    long long wide_tiles = 0, pair_tiles = 0, narrow_tiles = 0;
    for (int i = 0; i < n; ++i)
        if (groups[i].M > 0) {
            const GroupDesc &g = groups[i];
            all_n256 = all_n256 && (g.N % 256 == 0);
            all_n_ge256 = all_n_ge256 && (g.N >= 256);
            wide_tiles += (long long)((g.M + 127) / 128) * ((g.N + 255) / 256);
            pair_tiles += (long long)((g.M + 255) / 256) * ((g.N + 255) / 256);
            narrow_tiles += (long long)((g.M + 127) / 128) * ((g.N + 127) / 128);
        }
    if (forced >= 0 && forced < kNumKinds) {
        if (needs_n256(forced) && !all_n256)
            return kKindStream;
        // a pair's B scale load spans two 128-row blocks: N >= 256
        if (forced == kKindPair && !all_n_ge256)
            return kKindStream;
        // stream-K unit indices are 32-bit
        if (forced == kKindWideSK) {
            long long units = 0;
            for (int i = 0; i < n; ++i)
                if (groups[i].M > 0)
                    units += (long long)((groups[i].M + 127) / 128) * ((groups[i].N + 255) / 256) *
                             (groups[i].K / 256);
            if (units >= (1ll << 30))
                return kKindWide;
        }
        return forced;
    }
    const int pairs = sm_count / 2 > 0 ? sm_count / 2 : 1;
    const long long rounds_wide = (wide_tiles + sm_count - 1) / (sm_count > 0 ? sm_count : 1);
    const long long rounds_pair = (pair_tiles + pairs - 1) / pairs;
    // A call whose 128 x 128 tiles fit one round of the grid runs them: twice
    // the CTAs of 128 x 256 tiles, each with half the work (GEMM us, 128 x 128
    // against 128 x 256: 4 x [256, 2048, 2048] 7.8 / 10.2, 8 x [128, 1024,
    // 4096] 11.1 / 14.4, 6 x [300, 1024, 1024] 5.5 / 7.4, 2 x [M, 256, 256]
    // 3.7 / 5.3).  SwiGLU needs the 256-column tile.
    if (!need_bn256 && narrow_tiles <= sm_count)
        return kKindCompute;
    // CTA pairs whenever they need no more rounds of the grid than single
    // CTAs: each SM then stages half the B bytes (4096^3 groups 14 / 14
    // rounds; 2 x [512, 3072, 4096] 1 / 1, 14.0 against 14.3 us; 2 x [1000,
    // 4096, 2048] 2 / 2, 14.6 against 15.5 us), but not when padding M to 256
    // rows adds a round (the MoE shapes: gate/up 3 / 2, down 5 / 4; 8 x [64,
    // 4096, 7168] 2 / 1, 33.8 against 26.8 us)
    if (all_n_ge256 && rounds_pair <= rounds_wide)
        return kKindPair;
    return all_n256 ? kKindWide : kKindStream;
}

// L2 policy for B and its scales (0 normal, 1 evict_first, 2 evict_last;
// A and the A scales are always evict_last).  B is read once per M-tile of
// its group, by CTAs running side by side; keeping it (2) measured best in
// the bench's back-to-back steps: GEMM / step us, evict_last against
// normal, square 119.4-119.8 / 125.3 against 120.4 / 125.4, moe_gate_up
// 38.1-38.2 / 46.3-46.4 against 38.4 / 46.9, moe_down 27.2 / 32.6 against
// 27.2 / 33.0; evict_first was slower on every shape but the single-round
// one (square 123.3, moe_down 28.5 us).
int choose_b_policy()
{
    const int o = b_policy_override();
    return (o >= 0 && o <= 2) ? o : 2;
}

// L2 prefetch distance for B, in stages ahead of the MMAs; 0 (the default)
// leaves the prefetch warp idle.  Since the barrier waits sleep instead of
// polling, the loaders alone keep enough HBM reads in flight: measured with
// the prefetcher off / 2 / 6 / 10 stages ahead, moe_gate_up 38.3-38.6 /
// 39.3 / 41.2-41.4 / 41.9 us, moe_down 27.3-27.5 / 27.8 / 27.7-28.0 / 28.5,
// square and single-round calls unchanged.
int choose_prefetch()
{
    const int forced = env_int("NVFP4_PF_STAGES", -1);
    return forced >= 0 ? forced : 0;
}

// launches a call needs for tile width bn (one per 32 non-empty groups,
// more only past 2^30 tiles); must agree with plan_and_launch
int count_launches(const GroupDesc *groups, int num_groups, int bm, int bn)
{
    int launches = 0, in_launch = 0;
    long long tiles_in_launch = 0;
    for (int i = 0; i < num_groups; ++i) {
        const GroupDesc &g = groups[i];
        if (g.M == 0)
            continue;
        const long long tiles =
            (long long)((g.M + bm - 1) / bm) * (long long)((g.N + bn - 1) / bn);
        if (launches == 0 || in_launch == kMaxGroups || tiles_in_launch + tiles > kMaxTilesPerLaunch) {
            ++launches;
            in_launch = 0;
            tiles_in_launch = 0;
        }
        ++in_launch;
        tiles_in_launch += tiles;
    }
    return launches;
}

// Plan and launch a validated call.  `err_for_launch(l)` gives the status
// words of launch l.  Tensor maps of every launch are encoded before the
// first launch, so a rejected map launches nothing.  The parameter blocks
// live in a per-thread vector whose capacity is kept between calls.
template <class ErrFn>
int plan_and_launch(const GroupDesc *groups, int num_groups, cudaStream_t stream, int dev,
                    int sm_count, int kind, ErrFn err_for_launch, const GemmEpilogue *epi = nullptr,
                    const SkScratch *sk = nullptr, bool early_ab = false)
{
    const bool swiglu = epi && epi->swiglu;
    const bool out_bf16 = epi && epi->out_bf16;
    bool any_alpha = false;
    if (epi && epi->alpha)
        for (int i = 0; i < num_groups; ++i)
            any_alpha = any_alpha || epi->alpha[i] != 1.0f;
    const bool ex = swiglu || out_bf16 || any_alpha;
    static thread_local std::vector<KernelParams> plist;
    const KindInfo &ki = kind_info(kind);
    const int b_policy = choose_b_policy();
    const int pf = choose_prefetch();
    const unsigned long long timeout = wait_timeout_ns();
    const int drop = debug_drop_stage();
    const CUtensorMapSwizzle c_swizzle =
        ki.epi_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    plist.clear();
    int rc = NVFP4_OK;
    for (int i = 0; i < num_groups && rc == NVFP4_OK; ++i) {
        const GroupDesc &g = groups[i];
        if (g.M == 0)
            continue;
        const int grid_m = (g.M + ki.bm - 1) / ki.bm;
        const int grid_n = (g.N + ki.bn - 1) / ki.bn;
        const long long tiles = (long long)grid_m * grid_n;
        if (plist.empty() || plist.back().g.num_groups == kMaxGroups ||
            plist.back().g.total_tiles + tiles > kMaxTilesPerLaunch) {
            plist.emplace_back();
            std::memset(&plist.back(), 0, sizeof(KernelParams));
            GemmParams &P = plist.back().g;
            P.err = err_for_launch((int)plist.size() - 1);
            P.timeout_ns = timeout;
            P.b_policy = b_policy;
            P.pf_stages = pf;
            P.debug_drop_stage = drop;
            P.out_bf16 = out_bf16 ? 1 : 0;
            P.swiglu = swiglu ? 1 : 0;
            P.early_ab = early_ab ? 1 : 0;
            if (ki.sk) {
                P.sk_ws = sk->ws;
                P.sk_flags = sk->flags;
                P.sk_epoch = sk->epoch;
            }
        }
        KernelParams &PP = plist.back();
        GemmParams &P = PP.g;
        const int j = P.num_groups;
        rc = encode_map_operand(&P.tmA[j], g.A, (uint64_t)g.M, (uint64_t)g.K, kBM, ki.chunks);
        if (rc == NVFP4_OK)
            rc = encode_map_operand(&P.tmB[j], g.B, (uint64_t)g.N, (uint64_t)g.K, ki.box_b,
                                    ki.chunks);
        if (rc == NVFP4_OK)
            rc = encode_map_sf(&PP.tmSFA[j], g.SFA, (uint64_t)g.M, (uint64_t)g.K, ki.sf_atoms, 1);
        if (rc == NVFP4_OK)
            rc = encode_map_sf(&PP.tmSFB[j], g.SFB, (uint64_t)g.N, (uint64_t)g.K, ki.sf_atoms,
                               ki.sfb_blocks);
        const uint64_t n_out = swiglu ? (uint64_t)g.N / 2 : (uint64_t)g.N;
        const CUtensorMapDataType c_type =
            out_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        if (rc == NVFP4_OK)
            rc = encode_map_2d(&P.tmC[j], c_type, g.C, n_out, (uint64_t)g.M, n_out * 2, ki.epi_cols, 32,
                               c_swizzle);
        // the single-store form of a CTA's last tile, where C's rows are
        // whole 64-column blocks; otherwise (or if the driver declines the
        // map) the last tile takes the per-chunk stores
        P.c_wide[j] = 0;
        if (rc == NVFP4_OK && n_out % 64 == 0 &&
            encode_map_c_wide(&P.tmCw[j], c_type, g.C, (uint64_t)g.M, n_out,
                              (uint32_t)((swiglu ? ki.bn / 2 : ki.bn) / 64)) == NVFP4_OK)
            P.c_wide[j] = 1;
        P.alpha[j] = (epi && epi->alpha) ? epi->alpha[i] : 1.0f;
        P.M[j] = g.M;
        P.N[j] = g.N;
        P.kchunks[j] = g.K / kChunkK;
        P.grid_m[j] = grid_m;
        P.total_tiles += (int)tiles;
        P.tile_end[j] = P.total_tiles;
        if (ki.sk) {
            const int bk = ki.chunks * kChunkK;
            P.units_total += (int)tiles * ((g.K + bk - 1) / bk);
            P.unit_end[j] = P.units_total;
        }
        P.num_groups = j + 1;
    }
    for (size_t l = 0; l < plist.size() && rc == NVFP4_OK; ++l) {
        const KernelParams &P = plist[l];
        // stream-K: one range of units per SM (at least one unit each)
        const int grid = ki.sk ? (P.g.units_total < sm_count ? P.g.units_total : sm_count)
                               : grid_size(dev, kind, P.g.total_tiles, sm_count);
        if (ki.launch(P, grid, stream, ex) != cudaSuccess || cudaGetLastError() != cudaSuccess)
            rc = NVFP4_ERR_CUDA;
    }
    return rc;
}

// ---------------------------------------------------------------------------
// SWAP: the transposed product on CTA pairs (gemm_swap_kernel.cuh)
// ---------------------------------------------------------------------------

// Token tiles of a group of M rows: at most 256 rows each, starting at
// multiples of 128 rows (where the tiled scales start a new 128-row block);
// a remainder of 257..384 rows is split 128 + rest, so both tiles stay
// within 256 rows and as even as the 128-row grid allows.  Returns the tile
// count and writes the start rows (and, past the last, M) to starts.
int token_tiles(int M, int *starts, int cap)
{
    int n = 0, m = 0;
    while (m < M && n < cap) {
        const int rem = M - m;
        const int take = rem <= kSwapMaxTok ? rem : (rem <= kSwapMaxTok + 128 ? 128 : kSwapMaxTok);
        starts[n++] = m;
        m += take;
    }
    starts[n] = m;
    return m == M ? n : -1;
}

// number of token tiles token_tiles() makes for a group of M > 0 rows
int token_tile_count(int M)
{
    int n = 0, rem = M;
    while (rem > kSwapMaxTok + 128) {
        ++n;
        rem -= kSwapMaxTok;
    }
    return n + (rem > kSwapMaxTok ? 2 : 1);
}

// launches of a swap call: a new launch when either the group or the token
// tile table of the current one is full (a group's token tiles may continue
// in the next launch); must agree with plan_and_launch_swap
int count_launches_swap(const GroupDesc *groups, int num_groups)
{
    int launches = 0, nw = 0, nt = 0;
    for (int i = 0; i < num_groups; ++i) {
        const GroupDesc &g = groups[i];
        if (g.M == 0)
            continue;
        int left = token_tile_count(g.M);
        while (left > 0) {
            if (launches == 0 || nw == kSwapMaxW || nt == kSwapMaxT) {
                ++launches;
                nw = 0;
                nt = 0;
            }
            const int take = left < kSwapMaxT - nt ? left : kSwapMaxT - nt;
            ++nw;
            nt += take;
            left -= take;
        }
    }
    return launches;
}

// Plan and launch a validated call on the swap kernel: every group's token
// tiles, their tensor maps (offset pointers into A, the tiled SFA and C),
// the group's B maps, one parameter block per launch.  All maps are encoded
// before the first launch.
template <class ErrFn>
int plan_and_launch_swap(const GroupDesc *groups, int num_groups, cudaStream_t stream, int dev,
                         ErrFn err_for_launch, const GemmEpilogue *epi, bool early_ab)
{
    const bool out_bf16 = epi && epi->out_bf16;
    bool any_alpha = false;
    if (epi && epi->alpha)
        for (int i = 0; i < num_groups; ++i)
            any_alpha = any_alpha || epi->alpha[i] != 1.0f;
    const bool ex = out_bf16 || any_alpha;
    static thread_local std::vector<SwapParams> plist;
    static thread_local std::vector<int> starts;
    const CUtensorMapDataType c_type =
        out_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    plist.clear();
    int rc = NVFP4_OK;
    for (int i = 0; i < num_groups && rc == NVFP4_OK; ++i) {
        const GroupDesc &g = groups[i];
        if (g.M == 0)
            continue;
        starts.resize((size_t)token_tile_count(g.M) + 1);
        const int ntt = token_tiles(g.M, starts.data(), (int)starts.size() - 1);
        if (ntt != token_tile_count(g.M))
            return NVFP4_ERR_INVALID_ARGUMENT;
        const int wt = (g.N + CfgSwap::BW - 1) / CfgSwap::BW;
        int done = 0;
        while (done < ntt && rc == NVFP4_OK) {
            if (plist.empty() || plist.back().num_w == kSwapMaxW ||
                plist.back().num_w == 0 ||
                plist.back().w_tfirst[plist.back().num_w - 1] + plist.back().w_tcount[plist.back().num_w - 1] ==
                    kSwapMaxT) {
                plist.emplace_back();
                std::memset(&plist.back(), 0, sizeof(SwapParams));
                SwapParams &P = plist.back();
                P.err = err_for_launch((int)plist.size() - 1);
                P.timeout_ns = wait_timeout_ns();
                P.b_policy = choose_b_policy();
                P.pf_stages = choose_prefetch();
                P.debug_drop_stage = debug_drop_stage();
                P.out_bf16 = out_bf16 ? 1 : 0;
                P.early_ab = early_ab ? 1 : 0;
            }
            SwapParams &P = plist.back();
            const int w = P.num_w;
            const int t0 = w > 0 ? P.w_tfirst[w - 1] + P.w_tcount[w - 1] : 0;
            const int take = (ntt - done) < (kSwapMaxT - t0) ? (ntt - done) : (kSwapMaxT - t0);
            rc = encode_map_operand(&P.tmW[w], g.B, (uint64_t)g.N, (uint64_t)g.K, kBM, 1);
            if (rc == NVFP4_OK)
                rc = encode_map_sf(&P.tmSW[w], g.SFB, (uint64_t)g.N, (uint64_t)g.K, CfgSwap::kMmas, 1);
            for (int k = 0; k < take && rc == NVFP4_OK; ++k) {
                const int t = t0 + k;
                const int m0 = starts[done + k], mt = starts[done + k + 1] - m0;
                const int npad = (mt + 15) / 16 * 16;
                const int nsx = (mt + 127) / 128;
                const uint8_t *a = static_cast<const uint8_t *>(g.A) + (size_t)m0 * (size_t)(g.K / 2);
                const uint8_t *sa =
                    static_cast<const uint8_t *>(g.SFA) + (size_t)(m0 / 128) * (size_t)(g.K / 64) * 512u;
                uint8_t *c = static_cast<uint8_t *>(g.C) + (size_t)m0 * (size_t)g.N * 2u;
                rc = encode_map_operand(&P.tmX[t], a, (uint64_t)mt, (uint64_t)g.K, (uint32_t)(npad / 2), 1);
                if (rc == NVFP4_OK)
                    rc = encode_map_sf(&P.tmSX[t], sa, (uint64_t)mt, (uint64_t)g.K, CfgSwap::kMmas, (uint32_t)nsx);
                if (rc == NVFP4_OK)
                    rc = encode_map_2d(&P.tmC[t], c_type, c, (uint64_t)g.N, (uint64_t)mt, (uint64_t)g.N * 2, 32, 32,
                                       CU_TENSOR_MAP_SWIZZLE_NONE);
                P.t_group[t] = w;
                P.t_rows[t] = mt;
                P.t_npad[t] = npad;
                P.t_sfx[t] = nsx;
            }
            P.w_N[w] = g.N;
            P.w_kchunks[w] = g.K / kChunkK;
            P.w_tiles[w] = wt;
            P.w_tfirst[w] = t0;
            P.w_tcount[w] = take;
            P.alpha[w] = (epi && epi->alpha) ? epi->alpha[i] : 1.0f;
            P.total_tiles += wt * take;
            P.tile_end[w] = P.total_tiles;
            P.num_w = w + 1;
            done += take;
        }
    }
    for (size_t l = 0; l < plist.size() && rc == NVFP4_OK; ++l) {
        const SwapParams &P = plist[l];
        const int pairs = g_max_pairs[dev][kKindSwap];
        const int grid = 2 * (P.total_tiles < pairs ? P.total_tiles : pairs);
        LaunchCfg L;
        make_launch_cfg(L, grid, CfgSwap::kThreads, CfgSwap::kSmemBytes, true, stream);
        const cudaError_t e = ex ? cudaLaunchKernelEx(&L.cfg, nvfp4_group_gemm_swap_kernel<CfgSwap, true>, P)
                                 : cudaLaunchKernelEx(&L.cfg, nvfp4_group_gemm_swap_kernel<CfgSwap, false>, P);
        if (e != cudaSuccess || cudaGetLastError() != cudaSuccess)
            rc = NVFP4_ERR_CUDA;
    }
    return rc;
}

// launches of a call on `kind` (0: every group empty)
int launches_of(const GroupDesc *groups, int num_groups, int kind)
{
    if (kind == kKindSwap)
        return count_launches_swap(groups, num_groups);
    return count_launches(groups, num_groups, kind_info(kind).bm, kind_info(kind).bn);
}

// the launches of a validated call on `kind`
template <class ErrFn>
int dispatch(const GroupDesc *groups, int num_groups, cudaStream_t stream, int dev, int sm_count, int kind,
             ErrFn err_for_launch, const GemmEpilogue *epi = nullptr, const SkScratch *sk = nullptr,
             bool early_ab = false)
{
    if (kind == kKindSwap)
        return plan_and_launch_swap(groups, num_groups, stream, dev, err_for_launch, epi, early_ab);
    return plan_and_launch(groups, num_groups, stream, dev, sm_count, kind, err_for_launch, epi, sk, early_ab);
}

}  // namespace
}  // namespace nvfp4

extern "C" int nvfp4_group_gemm(const GroupDesc *groups, int num_groups, cudaStream_t stream)
{
    using namespace nvfp4;
    int rc = validate_call(groups, num_groups);
    if (rc != NVFP4_OK)
        return rc;
    DeviceState *dev = nullptr;
    rc = current_device(&dev);
    if (rc != NVFP4_OK)
        return rc;
    int kind = choose_kind(groups, num_groups, dev->sm_count);
    if (launches_of(groups, num_groups, kind) == 0)
        return NVFP4_OK;
    SkScratch sk{};
    if (kind == kKindWideSK && sk_scratch(stream, dev->sm_count, &sk) != NVFP4_OK)
        kind = kKindWide;
    int dev_id = 0;
    cudaGetDevice(&dev_id);
    rc = ensure_kernel_attributes(dev_id, kind);
    if (rc != NVFP4_OK)
        return rc;
    uint32_t *err = dev->err;
    return dispatch(groups, num_groups, stream, dev_id, dev->sm_count, kind,
                           [err](int) { return err; }, nullptr, &sk);
}

extern "C" int nvfp4_group_gemm_ex(const GroupDesc *groups, int num_groups, const GemmEpilogue *epi,
                                   cudaStream_t stream)
{
    using namespace nvfp4;
    int rc = validate_call(groups, num_groups);
    if (rc != NVFP4_OK)
        return rc;
    const bool swiglu = epi && epi->swiglu;
    if (swiglu)
        for (int i = 0; i < num_groups; ++i)
            if (groups[i].M > 0 && groups[i].N % 256 != 0)
                return NVFP4_ERR_INVALID_ARGUMENT;
    DeviceState *dev = nullptr;
    rc = current_device(&dev);
    if (rc != NVFP4_OK)
        return rc;
    int kind = choose_kind(groups, num_groups, dev->sm_count, swiglu);
    if (launches_of(groups, num_groups, kind) == 0)
        return NVFP4_OK;
    SkScratch sk{};
    if (kind == kKindWideSK && sk_scratch(stream, dev->sm_count, &sk) != NVFP4_OK)
        kind = kKindWide;
    int dev_id = 0;
    cudaGetDevice(&dev_id);
    rc = ensure_kernel_attributes(dev_id, kind);
    if (rc != NVFP4_OK)
        return rc;
    uint32_t *err = dev->err;
    return dispatch(groups, num_groups, stream, dev_id, dev->sm_count, kind,
                           [err](int) { return err; }, epi, &sk);
}

// ---------------------------------------------------------------------------
// nvfp4_relayout_and_gemm: the scale relayout of every group and the grouped
// GEMM as one call.  The GEMM follows the relayout in the stream with a
// programmatic launch, and since the library launched that relayout itself
// it knows A and B were complete before it began: the GEMM's A and B loads
// start without waiting for the relayout to finish (early_ab); only the
// scale loads, the MMAs and the epilogue wait for it.
// ---------------------------------------------------------------------------
extern "C" int nvfp4_relayout_and_gemm(const StepDesc *steps, int num_groups, const GemmEpilogue *epi,
                                       cudaStream_t stream)
{
    using namespace nvfp4;
    if (!steps || num_groups < 1)
        return NVFP4_ERR_INVALID_ARGUMENT;
    if (num_groups > kMaxGroupsPerCall)
        return NVFP4_ERR_TOO_MANY;
    static thread_local std::vector<GroupDesc> groups;
    static thread_local std::vector<SfRelayoutDesc> rel;
    groups.resize((size_t)num_groups);
    rel.clear();
    for (int i = 0; i < num_groups; ++i) {
        const StepDesc &s = steps[i];
        groups[i] = GroupDesc{s.A, s.B, s.SFA_tiled, s.SFB_tiled, s.C, s.M, s.N, s.K};
        if (s.M > 0) {
            if (!s.SFA || !s.SFB)
                return NVFP4_ERR_INVALID_ARGUMENT;
            if (!aligned16(s.SFA) || !aligned16(s.SFB))
                return NVFP4_ERR_MISALIGNED;
            rel.push_back(SfRelayoutDesc{s.SFA, s.SFA_tiled, s.M, s.K});
            rel.push_back(SfRelayoutDesc{s.SFB, s.SFB_tiled, s.N, s.K});
        }
    }
    int rc = validate_call(groups.data(), num_groups);
    if (rc != NVFP4_OK)
        return rc;
    const bool swiglu = epi && epi->swiglu;
    if (swiglu)
        for (int i = 0; i < num_groups; ++i)
            if (groups[i].M > 0 && groups[i].N % 256 != 0)
                return NVFP4_ERR_INVALID_ARGUMENT;
    DeviceState *dev = nullptr;
    rc = current_device(&dev);
    if (rc != NVFP4_OK)
        return rc;
    int kind = choose_kind(groups.data(), num_groups, dev->sm_count, swiglu);
    if (launches_of(groups.data(), num_groups, kind) == 0)
        return NVFP4_OK;
    SkScratch sk{};
    if (kind == kKindWideSK && sk_scratch(stream, dev->sm_count, &sk) != NVFP4_OK)
        kind = kKindWide;
    int dev_id = 0;
    cudaGetDevice(&dev_id);
    rc = ensure_kernel_attributes(dev_id, kind);
    if (rc != NVFP4_OK)
        return rc;
    rc = nvfp4_sf_relayout_group(rel.data(), (int)rel.size(), stream);
    if (rc != NVFP4_OK)
        return rc;
    uint32_t *err = dev->err;
    return dispatch(groups.data(), num_groups, stream, dev_id, dev->sm_count, kind,
                           [err](int) { return err; }, epi, &sk, true);
}

extern "C" int nvfp4_group_gemm_plan_for(const GroupDesc *groups, int num_groups, int sm_count,
                                         int *kind, int *launches)
{
    using namespace nvfp4;
    if (!kind || !launches || sm_count < 2)
        return NVFP4_ERR_INVALID_ARGUMENT;
    const int rc = validate_call(groups, num_groups);
    if (rc != NVFP4_OK)
        return rc;
    const int k = choose_kind(groups, num_groups, sm_count);
    *kind = k;
    *launches = launches_of(groups, num_groups, k);
    return NVFP4_OK;
}

extern "C" int nvfp4_group_gemm_plan(const GroupDesc *groups, int num_groups, int *kind,
                                     int *launches)
{
    using namespace nvfp4;
    if (!kind || !launches)
        return NVFP4_ERR_INVALID_ARGUMENT;
    int rc = validate_call(groups, num_groups);
    if (rc != NVFP4_OK)
        return rc;
    DeviceState *dev = nullptr;
    rc = current_device(&dev);
    if (rc != NVFP4_OK)
        return rc;
    return nvfp4_group_gemm_plan_for(groups, num_groups, dev->sm_count, kind, launches);
}

// ---------------------------------------------------------------------------
// nvfp4_group_gemm_noalloc: the same grouped GEMM for callers that may not
// allocate device memory at all.
//
// The kernel's only scratch is its status record (error bits and the first
// expired wait, two 32-bit words per launch).  nvfp4_group_gemm keeps that
// record in a word it allocates on first use; this entry point keeps it in
// the file-scope array below instead, which lives in the library's own
// module: every GPU that loads the library holds these 256 bytes until the
// process exits.
// ---------------------------------------------------------------------------
namespace nvfp4 {
namespace {

constexpr int kNoAllocScratchWords = 64;                    // 256 bytes
constexpr int kNoAllocMaxLaunches = kNoAllocScratchWords / 2;

static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchWords];

struct NoAllocDevice {
    bool ready;
    int sm_count;
    uint32_t *scratch;  // device address of g_noalloc_scratch on this device
};
std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_dev[kMaxDevices];

// One-time set-up for the current device (the first call on each device):
// capability check and the device address of the static scratch array.
// Neither allocates.
int noalloc_device(NoAllocDevice **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return NVFP4_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    NoAllocDevice &d = g_noalloc_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        if (!(major == 10 && minor == 3))
            return NVFP4_ERR_UNSUPPORTED;
        uint32_t *ptr = nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&ptr), g_noalloc_scratch) != cudaSuccess ||
            ptr == nullptr)
            return NVFP4_ERR_CUDA;
        d.sm_count = sms;
        d.scratch = ptr;
        d.ready = true;
    }
    *out = &d;
    return NVFP4_OK;
}

}  // namespace
}  // namespace nvfp4

extern "C" int nvfp4_group_gemm_noalloc(const GroupDesc *groups, int num_groups,
                                        cudaStream_t stream)
{
    using namespace nvfp4;
    int rc = validate_call(groups, num_groups);
    if (rc != NVFP4_OK)
        return rc;
    NoAllocDevice *dev = nullptr;
    rc = noalloc_device(&dev);
    if (rc != NVFP4_OK)
        return rc;
    // no stream-K here: its partial sums need allocated scratch
    int kind = choose_kind(groups, num_groups, dev->sm_count);
    if (kind == kKindWideSK)
        kind = kKindWide;
    // each launch needs its own two status words of the static scratch
    const int launches = launches_of(groups, num_groups, kind);
    if (launches == 0)
        return NVFP4_OK;
    if (launches > kNoAllocMaxLaunches)
        return NVFP4_ERR_TOO_MANY;   // more than 32 launches' worth (> 1024 non-empty groups)
    int dev_id = 0;
    cudaGetDevice(&dev_id);
    rc = ensure_kernel_attributes(dev_id, kind);
    if (rc != NVFP4_OK)
        return rc;
    // the status words must start at zero; the array keeps the previous
    // call's contents otherwise
    if (cudaMemsetAsync(dev->scratch, 0, sizeof(uint32_t) * 2 * launches, stream) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    uint32_t *scratch = dev->scratch;
    return dispatch(groups, num_groups, stream, dev_id, dev->sm_count, kind,
                           [scratch](int l) { return scratch + 2 * l; });
}
