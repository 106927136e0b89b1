// group_gemm.cu -- C-ABI entry point nvfp4_group_gemm: validation, the
// per-call tile plan, tensor maps and the launch of the persistent kernel.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/nvfp4_group_gemm.h"
#include "gemm_kernel.cuh"
#include "runtime.h"

namespace nvfp4 {
namespace {

constexpr int kBN = 128;
constexpr int kMaxDim = 1 << 20;
constexpr int kMaxGroupsPerCall = 4096;
constexpr long long kMaxTilesPerLaunch = 1ll << 30;

std::mutex g_attr_mu;
bool g_attr_set[64];

int ensure_kernel_attributes(int dev)
{
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (dev < 0 || dev >= 64)
        return NVFP4_ERR_UNSUPPORTED;
    if (!g_attr_set[dev]) {
        if (cudaFuncSetAttribute(nvfp4_group_gemm_kernel<kBN>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 GemmConfig<kBN>::kSmemBytes) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        g_attr_set[dev] = true;
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

// L2 policy for B and its scales: B is streamed once per M-tile of its
// group, and the M-tiles of one B strip run side by side, so the default
// keeps B at normal priority (A and the A scales are kept: evict_last)
int choose_b_policy()
{
    const int o = b_policy_override();
    return (o >= 0 && o <= 2) ? o : 0;
}

int launch_chunk(GemmParams &P, int sm_count, cudaStream_t stream)
{
    if (P.total_tiles == 0)
        return NVFP4_OK;
    const int grid = P.total_tiles < sm_count ? P.total_tiles : sm_count;
    nvfp4_group_gemm_kernel<kBN><<<grid, kThreads, GemmConfig<kBN>::kSmemBytes, stream>>>(P);
    return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // namespace
}  // namespace nvfp4

extern "C" int nvfp4_group_gemm(const GroupDesc *groups, int num_groups, cudaStream_t stream)
{
    using namespace nvfp4;
    if (!groups || num_groups < 1)
        return NVFP4_ERR_INVALID_ARGUMENT;
    if (num_groups > kMaxGroupsPerCall)
        return NVFP4_ERR_TOO_MANY;
    for (int i = 0; i < num_groups; ++i) {
        int rc = validate_group(groups[i]);
        if (rc != NVFP4_OK)
            return rc;
    }
    DeviceState *dev = nullptr;
    int rc = current_device(&dev);
    if (rc != NVFP4_OK)
        return rc;
    int dev_id = 0;
    cudaGetDevice(&dev_id);
    rc = ensure_kernel_attributes(dev_id);
    if (rc != NVFP4_OK)
        return rc;

    // Encode every tensor map before the first launch so that a rejected
    // map launches nothing.  Up to kMaxGroups non-empty groups share one
    // launch; a call with more is split into several launches on `stream`.
    // The parameter blocks live in a per-thread vector whose capacity is
    // kept, so steady-state calls allocate nothing.
    static thread_local std::vector<GemmParams> plist;
    const int b_policy = choose_b_policy();
    const unsigned long long timeout = wait_timeout_ns();
    const int drop = debug_drop_stage();
    auto fresh = [&]() -> GemmParams & {
        plist.emplace_back();
        GemmParams &P = plist.back();
        std::memset(&P, 0, sizeof(P));
        P.err = dev->err;
        P.timeout_ns = timeout;
        P.b_policy = b_policy;
        P.debug_drop_stage = drop;
        return P;
    };
    plist.clear();
    for (int i = 0; i < num_groups && rc == NVFP4_OK; ++i) {
        const GroupDesc &g = groups[i];
        if (g.M == 0)
            continue;
        const int grid_m = (g.M + kBM - 1) / kBM;
        const int grid_n = (g.N + kBN - 1) / kBN;
        const long long tiles = (long long)grid_m * grid_n;
        if (plist.empty() || plist.back().num_groups == kMaxGroups ||
            plist.back().total_tiles + tiles > kMaxTilesPerLaunch)
            fresh();
        GemmParams *P = &plist.back();
        const int j = P->num_groups;
        const uint64_t kbytes = (uint64_t)g.K / 2;
        rc = encode_map_2d(&P->tmA[j], CU_TENSOR_MAP_DATA_TYPE_UINT8, g.A, kbytes, (uint64_t)g.M,
                           kbytes, kBK / 2, kBM);
        if (rc == NVFP4_OK)
            rc = encode_map_2d(&P->tmB[j], CU_TENSOR_MAP_DATA_TYPE_UINT8, g.B, kbytes,
                               (uint64_t)g.N, kbytes, kBK / 2, kBN);
        if (rc == NVFP4_OK)
            rc = encode_map_2d(&P->tmC[j], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, g.C, (uint64_t)g.N,
                               (uint64_t)g.M, (uint64_t)g.N * 2, 64, 32);
        P->sfa[j] = static_cast<const uint8_t *>(g.SFA);
        P->sfb[j] = static_cast<const uint8_t *>(g.SFB);
        P->M[j] = g.M;
        P->N[j] = g.N;
        P->kiters[j] = g.K / kBK;
        P->grid_m[j] = grid_m;
        P->total_tiles += (int)tiles;
        P->tile_end[j] = P->total_tiles;
        P->num_groups = j + 1;
    }
    for (size_t l = 0; l < plist.size() && rc == NVFP4_OK; ++l)
        rc = launch_chunk(plist[l], dev->sm_count, stream);
    return rc;
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
NoAllocDevice g_noalloc_dev[64];

// One-time set-up for the current device (the first call on each device):
// capability check, the kernel's shared-memory attribute and the device
// address of the static scratch array.  None of these allocates.
int noalloc_device(NoAllocDevice **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (dev < 0 || dev >= 64)
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
        int rc = ensure_kernel_attributes(dev);
        if (rc != NVFP4_OK)
            return rc;
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
    if (!groups || num_groups < 1)
        return NVFP4_ERR_INVALID_ARGUMENT;
    if (num_groups > kMaxGroupsPerCall)
        return NVFP4_ERR_TOO_MANY;
    // pass 1: validate, and count the launches (each needs its own two
    // status words of the static scratch)
    int launches = 0, in_launch = 0;
    long long tiles_in_launch = 0;
    for (int i = 0; i < num_groups; ++i) {
        int rc = validate_group(groups[i]);
        if (rc != NVFP4_OK)
            return rc;
        const GroupDesc &g = groups[i];
        if (g.M == 0)
            continue;
        const long long tiles =
            (long long)((g.M + kBM - 1) / kBM) * (long long)((g.N + kBN - 1) / kBN);
        if (launches == 0 || in_launch == kMaxGroups || tiles_in_launch + tiles > kMaxTilesPerLaunch) {
            ++launches;
            in_launch = 0;
            tiles_in_launch = 0;
        }
        ++in_launch;
        tiles_in_launch += tiles;
    }
    if (launches == 0)
        return NVFP4_OK;
    if (launches > kNoAllocMaxLaunches)
        return NVFP4_ERR_TOO_MANY;   // more than 32 launches' worth (> 1024 non-empty groups)

    NoAllocDevice *dev = nullptr;
    int rc = noalloc_device(&dev);
    if (rc != NVFP4_OK)
        return rc;
    // the status words must start at zero; the array keeps the previous
    // call's contents otherwise
    if (cudaMemsetAsync(dev->scratch, 0, sizeof(uint32_t) * 2 * launches, stream) != cudaSuccess)
        return NVFP4_ERR_CUDA;

    // pass 2: one parameter block at a time (launch copies it), launched as
    // soon as its groups are encoded
    static thread_local GemmParams P;
    const int b_policy = choose_b_policy();
    const unsigned long long timeout = wait_timeout_ns();
    const int drop = debug_drop_stage();
    int launch = 0;
    bool open = false;
    for (int i = 0; i < num_groups && rc == NVFP4_OK; ++i) {
        const GroupDesc &g = groups[i];
        if (g.M == 0)
            continue;
        const int grid_m = (g.M + kBM - 1) / kBM;
        const int grid_n = (g.N + kBN - 1) / kBN;
        const long long tiles = (long long)grid_m * grid_n;
        if (open && (P.num_groups == kMaxGroups || P.total_tiles + tiles > kMaxTilesPerLaunch)) {
            rc = launch_chunk(P, dev->sm_count, stream);
            open = false;
            ++launch;
            if (rc != NVFP4_OK)
                break;
        }
        if (!open) {
            std::memset(&P, 0, sizeof(P));
            P.err = dev->scratch + 2 * launch;
            P.timeout_ns = timeout;
            P.b_policy = b_policy;
            P.debug_drop_stage = drop;
            open = true;
        }
        const int j = P.num_groups;
        const uint64_t kbytes = (uint64_t)g.K / 2;
        rc = encode_map_2d(&P.tmA[j], CU_TENSOR_MAP_DATA_TYPE_UINT8, g.A, kbytes, (uint64_t)g.M,
                           kbytes, kBK / 2, kBM);
        if (rc == NVFP4_OK)
            rc = encode_map_2d(&P.tmB[j], CU_TENSOR_MAP_DATA_TYPE_UINT8, g.B, kbytes,
                               (uint64_t)g.N, kbytes, kBK / 2, kBN);
        if (rc == NVFP4_OK)
            rc = encode_map_2d(&P.tmC[j], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, g.C, (uint64_t)g.N,
                               (uint64_t)g.M, (uint64_t)g.N * 2, 64, 32);
        P.sfa[j] = static_cast<const uint8_t *>(g.SFA);
        P.sfb[j] = static_cast<const uint8_t *>(g.SFB);
        P.M[j] = g.M;
        P.N[j] = g.N;
        P.kiters[j] = g.K / kBK;
        P.grid_m[j] = grid_m;
        P.total_tiles += (int)tiles;
        P.tile_end[j] = P.total_tiles;
        P.num_groups = j + 1;
    }
    if (rc == NVFP4_OK && open)
        rc = launch_chunk(P, dev->sm_count, stream);
    return rc;
}
