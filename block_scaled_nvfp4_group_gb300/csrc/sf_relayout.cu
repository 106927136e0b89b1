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
// The relayout is a byte permutation, HBM-bound: one CTA moves up to four
// 128-row x 64-scale blocks (32 KiB in, 32 KiB out) through shared memory,
// with 16-byte loads along source rows (all issued before the first wait) and
// 16-byte stores along atom rows, both coalesced.  Algorithmic traffic: rows * K/16 bytes read, the tiled size
// written.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/nvfp4_group_gemm.h"
#include "ptx.cuh"
#include "runtime.h"

namespace nvfp4 {
namespace {

constexpr int kMaxDescs = 64;     // relayouts per launch (param block)
constexpr int kChunkScales = 64;  // scale columns per CTA = 16 atoms
constexpr int kRowBlocks = 4;     // 128-row blocks per CTA
constexpr int kThreads = 256;
constexpr int kPitchWords = 17;   // 64 bytes + 4 bytes pad per staged row
constexpr int kMaxDim = 1 << 20;
constexpr int kMaxCount = 4096;
// 16-byte loads per thread: kRowBlocks * 128 rows * 4 vectors / kThreads
constexpr int kLoadsPerThread = kRowBlocks * 128 * (kChunkScales / 16) / kThreads;

struct RelayoutParams {
    const uint8_t *src[kMaxDescs];
    uint8_t *dst[kMaxDescs];
    int rows[kMaxDescs];
    int kcols[kMaxDescs];     // K / 16 scale columns per row
    int chunks[kMaxDescs];    // ceil(kcols / 64)
    int item_end[kMaxDescs];  // inclusive prefix sum of row-block groups * chunks
    int count;
};

// One CTA: kRowBlocks consecutive 128-row blocks x one 64-column chunk.
// Every thread issues all of its 16-byte loads before the first shared store,
// so a CTA keeps up to 32 KiB of reads in flight.
__global__ void __launch_bounds__(kThreads) sf_relayout_kernel(const __grid_constant__ RelayoutParams p)
{
    __shared__ uint32_t tile[kRowBlocks * 128 * kPitchWords];
    // programmatic launch: start early, but read and write global memory only
    // once the previous kernel in the stream is done
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();

    const int item = blockIdx.x;
    int d = 0;
    while (item >= p.item_end[d])
        ++d;
    const int local = item - (d > 0 ? p.item_end[d - 1] : 0);
    const int chunks = p.chunks[d];
    const int rbg = local / chunks;             // group of kRowBlocks row blocks
    const int kc = local % chunks;
    const int kcols = p.kcols[d];
    const int rows = p.rows[d];
    const int rblocks = (rows + 127) / 128;
    const int nrb = min(kRowBlocks, rblocks - rbg * kRowBlocks);   // row blocks here
    const int width = min(kChunkScales, kcols - kc * kChunkScales);  // multiple of 16
    const int nvec = width / 16;
    const int row0 = rbg * kRowBlocks * 128;

    // loads: rows [row0, row0 + nrb*128) x `width` bytes, zero past `rows`
    const uint8_t *src = p.src[d] + (size_t)kc * kChunkScales;
    const int nload = nrb * 128 * nvec;
    uint4 x[kLoadsPerThread];
#pragma unroll
    for (int i = 0; i < kLoadsPerThread; ++i) {
        const int v = threadIdx.x + i * kThreads;
        const int r = v / nvec, c = v % nvec;
        x[i] = make_uint4(0u, 0u, 0u, 0u);
        if (v < nload && row0 + r < rows)
            x[i] = __ldcs(reinterpret_cast<const uint4 *>(src + (size_t)(row0 + r) * kcols) + c);
    }
#pragma unroll
    for (int i = 0; i < kLoadsPerThread; ++i) {
        const int v = threadIdx.x + i * kThreads;
        if (v < nload) {
            const int r = v / nvec, c = v % nvec;
            uint32_t *t = tile + r * kPitchWords + c * 4;
            t[0] = x[i].x;
            t[1] = x[i].y;
            t[2] = x[i].z;
            t[3] = x[i].w;
        }
    }
    __syncthreads();

    // atom a of row block rr: 16-byte row q holds rows q, q+32, q+64, q+96
    const int natoms = width / 4;
    const int nout = nrb * natoms * 32;
    for (int o = threadIdx.x; o < nout; o += kThreads) {
        const int rr = o / (natoms * 32);
        const int a = (o >> 5) % natoms, q = o & 31;
        const uint32_t *t = tile + rr * 128 * kPitchWords;
        uint4 y;
        y.x = t[(q)*kPitchWords + a];
        y.y = t[(q + 32) * kPitchWords + a];
        y.z = t[(q + 64) * kPitchWords + a];
        y.w = t[(q + 96) * kPitchWords + a];
        const size_t rb = (size_t)rbg * kRowBlocks + rr;
        uint8_t *dst = p.dst[d] + (rb * (kcols / 4) + (size_t)kc * (kChunkScales / 4) + a) * 512;
        *reinterpret_cast<uint4 *>(dst + q * 16) = y;
    }
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

    RelayoutParams P{};
    auto launch = [&]() -> int {
        if (P.count == 0)
            return NVFP4_OK;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(P.item_end[P.count - 1]);
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
    int items = 0;
    for (int i = 0; i < count; ++i) {
        const SfRelayoutDesc &d = descs[i];
        if (d.rows == 0)
            continue;
        const int kcols = d.K / 16;
        const int chunks = (kcols + kChunkScales - 1) / kChunkScales;
        const int rblocks = (d.rows + 127) / 128;
        const long long n = (long long)((rblocks + kRowBlocks - 1) / kRowBlocks) * chunks;
        if (P.count == kMaxDescs || (long long)items + n > (1ll << 30)) {
            rc = launch();
            if (rc != NVFP4_OK)
                return rc;
            P.count = 0;
            items = 0;
        }
        const int j = P.count++;
        P.src[j] = static_cast<const uint8_t *>(d.src);
        P.dst[j] = static_cast<uint8_t *>(d.dst);
        P.rows[j] = d.rows;
        P.kcols[j] = kcols;
        P.chunks[j] = chunks;
        items += (int)n;
        P.item_end[j] = items;
    }
    return launch();
}

int nvfp4_sf_relayout(const void *src, void *dst, int rows, int K, cudaStream_t stream)
{
    const SfRelayoutDesc d{src, dst, rows, K};
    return nvfp4_sf_relayout_group(&d, 1, stream);
}

}  // extern "C"
