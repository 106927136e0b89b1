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
// The relayout is a byte permutation, HBM-bound: one CTA moves a
// 128-row x 64-scale block (8 KiB in, 8 KiB out) through shared memory, with
// 16-byte loads along source rows and 16-byte stores along atom rows, both
// coalesced.  Algorithmic traffic: rows * K/16 bytes read, the tiled size
// written.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/nvfp4_group_gemm.h"
#include "runtime.h"

namespace nvfp4 {
namespace {

constexpr int kMaxDescs = 64;     // relayouts per launch (param block)
constexpr int kChunkScales = 64;  // scale columns per CTA = 16 atoms
constexpr int kThreads = 256;
constexpr int kPitchWords = 17;   // 64 bytes + 4 bytes pad per staged row
constexpr int kMaxDim = 1 << 20;
constexpr int kMaxCount = 4096;

struct RelayoutParams {
    const uint8_t *src[kMaxDescs];
    uint8_t *dst[kMaxDescs];
    int rows[kMaxDescs];
    int kcols[kMaxDescs];     // K / 16 scale columns per row
    int chunks[kMaxDescs];    // ceil(kcols / 64)
    int item_end[kMaxDescs];  // inclusive prefix sum of row blocks * chunks
    int count;
};

__global__ void __launch_bounds__(kThreads) sf_relayout_kernel(const __grid_constant__ RelayoutParams p)
{
    __shared__ uint32_t tile[128 * kPitchWords];

    const int item = blockIdx.x;
    int d = 0;
    while (item >= p.item_end[d])
        ++d;
    const int local = item - (d > 0 ? p.item_end[d - 1] : 0);
    const int chunks = p.chunks[d];
    const int rb = local / chunks;
    const int kc = local % chunks;
    const int kcols = p.kcols[d];
    const int rows = p.rows[d];
    const int width = min(kChunkScales, kcols - kc * kChunkScales);  // multiple of 16
    const int nvec = width / 16;

    // stage 128 rows x `width` scale bytes, zero past the last row
    const uint8_t *src = p.src[d] + (size_t)kc * kChunkScales;
    for (int v = threadIdx.x; v < 128 * nvec; v += kThreads) {
        const int r = v / nvec, c = v % nvec;
        const int grow = rb * 128 + r;
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (grow < rows)
            x = __ldcs(reinterpret_cast<const uint4 *>(src + (size_t)grow * kcols) + c);
        uint32_t *t = tile + r * kPitchWords + c * 4;
        t[0] = x.x;
        t[1] = x.y;
        t[2] = x.z;
        t[3] = x.w;
    }
    __syncthreads();

    // atom a of this chunk: 16-byte row q holds rows q, q+32, q+64, q+96
    const int natoms = width / 4;
    uint8_t *dst = p.dst[d] + ((size_t)rb * (kcols / 4) + (size_t)kc * (kChunkScales / 4)) * 512;
    for (int o = threadIdx.x; o < natoms * 32; o += kThreads) {
        const int a = o >> 5, q = o & 31;
        uint4 y;
        y.x = tile[(q)*kPitchWords + a];
        y.y = tile[(q + 32) * kPitchWords + a];
        y.z = tile[(q + 64) * kPitchWords + a];
        y.w = tile[(q + 96) * kPitchWords + a];
        *reinterpret_cast<uint4 *>(dst + (size_t)a * 512 + q * 16) = y;
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
        sf_relayout_kernel<<<P.item_end[P.count - 1], kThreads, 0, stream>>>(P);
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
        const long long n = (long long)((d.rows + 127) / 128) * chunks;
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
