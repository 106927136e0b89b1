// sf_relayout.cu -- scale-factor relayout kernel and its C-ABI entry points
// (nvfp4_sf_relayout, nvfp4_sf_relayout_group, nvfp4_sf_tiled_bytes).
//
// Plain row-major E4M3FN scales [rows][K/16] become 512-byte atoms, one per
// (128-row block rb, 64-element K block kb), stored [rb][kb] (kernelbot
// nvfp4-group-gemm submission 474067, TMA producer warp: scale source
// base + ((off_m/128) * (K/64) + off_k/64) * 512).  Inside an atom, the four
// scales of row r and K block kb sit at byte (r % 32) * 16 + (r / 32) * 4,
// the 32 x 16-byte shape of one tcgen05.cp 32x128b.warpx4 (474067,
// tcgen05_cp_nvfp4).  Rows past `rows` in the last block become zero.
//
// The relayout is a byte permutation, HBM-bound, done entirely in
// registers.  A warp takes 4 atom rows l (0..31) x 8 blocks of 16 scale
// columns (4 atoms each) of one 128-row block: lane = 8 (l % 4) + block.
// Each thread makes four 16-byte loads, rows l, l+32, l+64, l+96 of its
// column block (a warp instruction reads four rows x 128 contiguous bytes),
// transposes the 4 x 4 words in registers, and makes four 16-byte stores:
// row l of each of its four atoms (a warp instruction writes eight atoms x
// 64 contiguous bytes).  The warps of a CTA take neighbouring column groups
// of the same rows.  Small CTAs with few registers keep the whole call's
// loads in flight at once.  There is no shared memory and no wait to bound.
// Algorithmic traffic: rows * K/16 bytes read, the tiled size written.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/nvfp4_group_gemm.h"
#include "ptx.cuh"
#include "runtime.h"

namespace nvfp4 {
namespace {

constexpr int kMaxDescs = 64;     // relayouts per launch (param block)
constexpr int kThreads = 128;     // four warps, one work unit each
constexpr int kMaxDim = 1 << 20;
constexpr int kMaxCount = 4096;

struct RelayoutParams {
    const uint8_t *src[kMaxDescs];
    uint8_t *dst[kMaxDescs];
    int rows[kMaxDescs];
    int kcols[kMaxDescs];        // K / 16 scale columns per row
    int cgroups[kMaxDescs];      // groups of 128 scale columns per row: ceil(kcols / 128)
    int unit_end[kMaxDescs];     // inclusive prefix sum of row blocks * 8 * cgroups
    int count;
    int total_units;
};

__device__ __forceinline__ void st_na_v4(void *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__global__ void __launch_bounds__(kThreads) sf_relayout_kernel(const __grid_constant__ RelayoutParams p)
{
    // programmatic launch: read and write global memory only once the
    // previous kernel in the stream is done
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int unit = (int)blockIdx.x * (kThreads / 32) + (int)(threadIdx.x >> 5);
    if (unit >= p.total_units)
        return;
    int d = 0;
    while (unit >= p.unit_end[d])
        ++d;
    const int local = unit - (d > 0 ? p.unit_end[d - 1] : 0);
    const int cgs = p.cgroups[d];
    const int rb = local / (8 * cgs);
    const int rem = local - rb * 8 * cgs;
    const int lg = rem / cgs;                   // atom rows 4 lg .. 4 lg + 3
    const int cg = rem - lg * cgs;              // column group (fastest: neighbouring warps)
    const int l = 4 * lg + (lane >> 3);
    const int cblk = 8 * cg + (lane & 7);      // block of 16 scale columns = atoms 4 cblk .. + 3
    const int kcols = p.kcols[d];
    if (cblk * 16 >= kcols)
        return;
    const int nrows = min(128, p.rows[d] - rb * 128);   // rows past it read as zero
    const uint8_t *src = p.src[d] + (size_t)rb * 128 * kcols + (size_t)cblk * 16;
    uint4 v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int r = l + 32 * q;
        v[q] = r < nrows ? __ldg(reinterpret_cast<const uint4 *>(src + (size_t)r * kcols)) : make_uint4(0, 0, 0, 0);
    }
    uint8_t *o = p.dst[d] + ((size_t)rb * (kcols / 4) + (size_t)(4 * cblk)) * 512 + l * 16;
    // stores that do not allocate in L1 (every byte is written once):
    // relayout 6.77 -> 6.58 us on the MoE gate/up scales, 6.03 -> 5.89 us on
    // the 4096^3 call, alternating runs on one box
    st_na_v4(o, v[0].x, v[1].x, v[2].x, v[3].x);
    st_na_v4(o + 512, v[0].y, v[1].y, v[2].y, v[3].y);
    st_na_v4(o + 1024, v[0].z, v[1].z, v[2].z, v[3].z);
    st_na_v4(o + 1536, v[0].w, v[1].w, v[2].w, v[3].w);
}

int validate(const SfRelayoutDesc &d)
{
    if (d.rows < 0 || d.rows > kMaxDim || d.K < 256 || d.K > kMaxDim || d.K % 256 != 0)
        return NVFP4_ERR_INVALID_ARGUMENT;
    if (d.rows == 0)
        return NVFP4_OK;
    if (!d.src || !d.dst)
        return NVFP4_ERR_INVALID_ARGUMENT;
    if (!aligned16(d.src) || !aligned16(d.dst))
        return NVFP4_ERR_MISALIGNED;
    return NVFP4_OK;
}

}  // namespace
}  // namespace nvfp4

extern "C" {

size_t nvfp4_sf_tiled_bytes(int rows, int K)
{
    if (rows <= 0 || K <= 0 || K % 64 != 0)
        return 0;
    return (size_t)((rows + 127) / 128) * (size_t)(K / 64) * 512u;
}

int nvfp4_sf_relayout_group(const SfRelayoutDesc *descs, int count, cudaStream_t stream)
{
    using namespace nvfp4;
    if (!descs || count < 1)
        return NVFP4_ERR_INVALID_ARGUMENT;
    if (count > kMaxCount)
        return NVFP4_ERR_TOO_MANY;
    for (int i = 0; i < count; ++i) {
        int rc = validate(descs[i]);
        if (rc != NVFP4_OK)
            return rc;
    }
    DeviceState *dev = nullptr;
    int rc = current_device(&dev);
    if (rc != NVFP4_OK)
        return rc;

    static thread_local RelayoutParams P;
    auto launch = [&]() -> int {
        if (P.count == 0)
            return NVFP4_OK;
        P.total_units = P.unit_end[P.count - 1];
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((P.total_units + kThreads / 32 - 1) / (kThreads / 32));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = env_int("NVFP4_PDL", 1) != 0;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, sf_relayout_kernel, P) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
    };
    P.count = 0;
    int units = 0;
    for (int i = 0; i < count; ++i) {
        const SfRelayoutDesc &d = descs[i];
        if (d.rows == 0)
            continue;
        const int kcols = d.K / 16;
        const int cgroups = (kcols + 127) / 128;
        const long long n = (long long)((d.rows + 127) / 128) * 8 * cgroups;
        if (P.count == kMaxDescs || (long long)units + n > (1ll << 30)) {
            rc = launch();
            if (rc != NVFP4_OK)
                return rc;
            P.count = 0;
            units = 0;
        }
        const int j = P.count;
        P.count = j + 1;
        P.src[j] = static_cast<const uint8_t *>(d.src);
        P.dst[j] = static_cast<uint8_t *>(d.dst);
        P.rows[j] = d.rows;
        P.kcols[j] = kcols;
        P.cgroups[j] = cgroups;
        units += (int)n;
        P.unit_end[j] = units;
    }
    return launch();
}

int nvfp4_sf_relayout(const void *src, void *dst, int rows, int K, cudaStream_t stream)
{
    const SfRelayoutDesc d{src, dst, rows, K};
    return nvfp4_sf_relayout_group(&d, 1, stream);
}

}  // extern "C"
