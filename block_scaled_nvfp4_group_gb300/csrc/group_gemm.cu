// group_gemm.cu -- C-ABI entry points nvfp4_group_gemm and
// nvfp4_group_gemm_noalloc: validation, the per-call tile plan, the kernel
// configuration for the shape class, tensor maps and the launches of the
// persistent kernel.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/nvfp4_group_gemm.h"
#include "gemm_kernel.cuh"
#include "runtime.h"

namespace nvfp4 {
namespace {

constexpr int kMaxDim = 1 << 20;
constexpr int kMaxGroupsPerCall = 4096;
constexpr long long kMaxTilesPerLaunch = 1ll << 30;
constexpr int kMaxDevices = 64;

enum Kind : int {
    kKindStream = 0,
    kKindWide = 1,
    kKindCompute = 2,
    kKindWide512 = 3,
    kKindWideP2 = 4,
    kKindWideP4 = 5,
    kNumKinds = 6
};

bool needs_n256(int kind)
{
    return kind == kKindWide || kind == kKindWide512 || kind == kKindWideP2 || kind == kKindWideP4;
}

// Launch with programmatic stream serialization (unless NVFP4_PDL=0): the
// kernel may start while the previous kernel in the stream finishes, and
// waits for it (griddepcontrol.wait) before touching global memory.
template <class Cfg>
cudaError_t launch_kind(const GemmParams &P, int grid, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(Cfg::kThreads);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = env_int("NVFP4_PDL", 1) != 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, nvfp4_group_gemm_kernel<Cfg>, P);
}

struct KindInfo {
    int bn;
    int chunks;     // 128-byte K chunks per row per stage
    int epi_cols;
    int smem;
    const void *fn;
    cudaError_t (*launch)(const GemmParams &, int, cudaStream_t);
};

template <class Cfg>
KindInfo make_kind()
{
    return KindInfo{Cfg::BN, Cfg::kChunks, Cfg::kEpiCols, Cfg::kSmemBytes,
                    reinterpret_cast<const void *>(&nvfp4_group_gemm_kernel<Cfg>), &launch_kind<Cfg>};
}

const KindInfo &kind_info(int k)
{
    static const KindInfo table[kNumKinds] = {make_kind<CfgStream>(),  make_kind<CfgWide>(),
                                              make_kind<CfgCompute>(), make_kind<CfgWide512>(),
                                              make_kind<CfgWideP2>(),  make_kind<CfgWideP4>()};
    return table[k];
}

std::mutex g_attr_mu;
bool g_attr_set[kMaxDevices][kNumKinds];

int ensure_kernel_attributes(int dev, int kind)
{
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (dev < 0 || dev >= kMaxDevices)
        return NVFP4_ERR_UNSUPPORTED;
    if (!g_attr_set[dev][kind]) {
        const KindInfo &ki = kind_info(kind);
        if (cudaFuncSetAttribute(ki.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ki.smem) !=
            cudaSuccess)
            return NVFP4_ERR_CUDA;
        g_attr_set[dev][kind] = true;
    }
    return NVFP4_OK;
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
// with 512-K stages (CfgStream).  NVFP4_GEMM_KIND overrides the choice.
int choose_kind(const GroupDesc *groups, int n)
{
    const int forced = env_int("NVFP4_GEMM_KIND", -1);
    bool all_n256 = true;
    for (int i = 0; i < n; ++i)
        if (groups[i].M > 0)
            all_n256 = all_n256 && (groups[i].N % 256 == 0);
    if (forced >= 0 && forced < kNumKinds)
        return (!needs_n256(forced) || all_n256) ? forced : kKindStream;
    return all_n256 ? kKindWide : kKindStream;
}

// L2 policy for B and its scales: B is streamed once per M-tile of its
// group, and the M-tiles of one B strip run side by side, so the default
// keeps B at normal priority (A and the A scales are kept: evict_last)
int choose_b_policy()
{
    const int o = b_policy_override();
    return (o >= 0 && o <= 2) ? o : 0;
}

// L2 prefetch distance for B, in stages ahead of the MMAs: 6 measured best
// on the MoE shapes (the ring holds 4 stages); 0 turns the prefetcher off
int choose_prefetch()
{
    const int forced = env_int("NVFP4_PF_STAGES", -1);
    return forced >= 0 ? forced : 6;
}

// launches a call needs for tile width bn (one per 32 non-empty groups,
// more only past 2^30 tiles); must agree with plan_and_launch
int count_launches(const GroupDesc *groups, int num_groups, int bn)
{
    int launches = 0, in_launch = 0;
    long long tiles_in_launch = 0;
    for (int i = 0; i < num_groups; ++i) {
        const GroupDesc &g = groups[i];
        if (g.M == 0)
            continue;
        const long long tiles =
            (long long)((g.M + kBM - 1) / kBM) * (long long)((g.N + bn - 1) / bn);
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
int plan_and_launch(const GroupDesc *groups, int num_groups, cudaStream_t stream, int sm_count,
                    int kind, ErrFn err_for_launch)
{
    static thread_local std::vector<GemmParams> plist;
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
        const int grid_m = (g.M + kBM - 1) / kBM;
        const int grid_n = (g.N + ki.bn - 1) / ki.bn;
        const long long tiles = (long long)grid_m * grid_n;
        if (plist.empty() || plist.back().num_groups == kMaxGroups ||
            plist.back().total_tiles + tiles > kMaxTilesPerLaunch) {
            plist.emplace_back();
            GemmParams &P = plist.back();
            std::memset(&P, 0, sizeof(P));
            P.err = err_for_launch((int)plist.size() - 1);
            P.timeout_ns = timeout;
            P.b_policy = b_policy;
            P.pf_stages = pf;
            P.debug_drop_stage = drop;
        }
        GemmParams &P = plist.back();
        const int j = P.num_groups;
        rc = encode_map_operand(&P.tmA[j], g.A, (uint64_t)g.M, (uint64_t)g.K, kBM, ki.chunks);
        if (rc == NVFP4_OK)
            rc = encode_map_operand(&P.tmB[j], g.B, (uint64_t)g.N, (uint64_t)g.K, ki.bn, ki.chunks);
        if (rc == NVFP4_OK)
            rc = encode_map_2d(&P.tmC[j], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, g.C, (uint64_t)g.N,
                               (uint64_t)g.M, (uint64_t)g.N * 2, ki.epi_cols, 32, c_swizzle);
        P.sfa[j] = static_cast<const uint8_t *>(g.SFA);
        P.sfb[j] = static_cast<const uint8_t *>(g.SFB);
        P.M[j] = g.M;
        P.N[j] = g.N;
        P.kchunks[j] = g.K / kChunkK;
        P.grid_m[j] = grid_m;
        P.total_tiles += (int)tiles;
        P.tile_end[j] = P.total_tiles;
        P.num_groups = j + 1;
    }
    for (size_t l = 0; l < plist.size() && rc == NVFP4_OK; ++l) {
        const GemmParams &P = plist[l];
        const int grid = P.total_tiles < sm_count ? P.total_tiles : sm_count;
        if (ki.launch(P, grid, stream) != cudaSuccess || cudaGetLastError() != cudaSuccess)
            rc = NVFP4_ERR_CUDA;
    }
    return rc;
}

}  // namespace
}  // namespace nvfp4

extern "C" int nvfp4_group_gemm(const GroupDesc *groups, int num_groups, cudaStream_t stream)
{
    using namespace nvfp4;
    int rc = validate_call(groups, num_groups);
    if (rc != NVFP4_OK)
        return rc;
    const int kind = choose_kind(groups, num_groups);
    if (count_launches(groups, num_groups, kind_info(kind).bn) == 0)
        return NVFP4_OK;
    DeviceState *dev = nullptr;
    rc = current_device(&dev);
    if (rc != NVFP4_OK)
        return rc;
    int dev_id = 0;
    cudaGetDevice(&dev_id);
    rc = ensure_kernel_attributes(dev_id, kind);
    if (rc != NVFP4_OK)
        return rc;
    uint32_t *err = dev->err;
    return plan_and_launch(groups, num_groups, stream, dev->sm_count, kind,
                           [err](int) { return err; });
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
    const int kind = choose_kind(groups, num_groups);
    // each launch needs its own two status words of the static scratch
    const int launches = count_launches(groups, num_groups, kind_info(kind).bn);
    if (launches == 0)
        return NVFP4_OK;
    if (launches > kNoAllocMaxLaunches)
        return NVFP4_ERR_TOO_MANY;   // more than 32 launches' worth (> 1024 non-empty groups)

    NoAllocDevice *dev = nullptr;
    rc = noalloc_device(&dev);
    if (rc != NVFP4_OK)
        return rc;
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
    return plan_and_launch(groups, num_groups, stream, dev->sm_count, kind,
                           [scratch](int l) { return scratch + 2 * l; });
}
