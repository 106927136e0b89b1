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
// The relayout is a byte permutation, HBM-bound.  Persistent CTAs (four per
// SM) walk the work items (one 128-row block x 64 scale columns = 16 atoms,
// 8 KiB) round robin; each keeps four items in flight: a 2-D TMA load brings
// the row-major tile into shared memory (rows past `rows` and columns past
// K/16 read as zero), 256 threads transpose it (each 16-byte atom row is
// four 4-byte words from rows q, q+32, q+64, q+96; the lane order makes the
// shared-memory reads conflict-free) and write 32-byte runs of atoms to
// global memory while the next tiles load.  Algorithmic traffic: rows * K/16
// bytes read, the tiled size written.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/nvfp4_group_gemm.h"
#include "ptx.cuh"
#include "runtime.h"

namespace nvfp4 {
namespace {

constexpr int kMaxDescs = 64;     // relayouts per launch (param block)
constexpr int kChunkScales = 64;  // scale columns per item = 16 atoms
constexpr int kThreads = 256;
constexpr int kBufs = 4;          // items in flight per CTA
constexpr int kTileBytes = 128 * kChunkScales;
constexpr int kCtasPerSm = 4;
constexpr int kMaxDim = 1 << 20;
constexpr int kMaxCount = 4096;

struct RelayoutParams {
    CUtensorMap tm[kMaxDescs];   // uint8 {K/16, rows}, box {64, 128}, no swizzle
    uint8_t *dst[kMaxDescs];
    int kcols[kMaxDescs];        // K / 16 scale columns per row
    int chunks[kMaxDescs];       // ceil(kcols / 64)
    int item_end[kMaxDescs];     // inclusive prefix sum of row blocks * chunks
    int count;
    int total_items;
    uint32_t *err;
    unsigned long long timeout_ns;
};

__device__ __forceinline__ void decode_item(const RelayoutParams &p, int item, int &d, int &rb, int &cc)
{
    d = 0;
    while (item >= p.item_end[d])
        ++d;
    const int local = item - (d > 0 ? p.item_end[d - 1] : 0);
    rb = local / p.chunks[d];
    cc = local % p.chunks[d];
}

__global__ void __launch_bounds__(kThreads) sf_relayout_kernel(const __grid_constant__ RelayoutParams p)
{
    __shared__ __align__(128) uint8_t tile[kBufs][kTileBytes];
    __shared__ __align__(8) uint64_t bars[kBufs];
    __shared__ int ok_flag;
    // programmatic launch: start early, but read and write global memory only
    // once the previous kernel in the stream is done
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();

    const uint32_t bar0 = ptx::smem_addr(&bars[0]);
    if (threadIdx.x == 0) {
        for (int b = 0; b < kBufs; ++b)
            ptx::mbar_init(bar0 + 8u * b, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    const uint64_t pol = ptx::policy_evict_first();
    uint32_t inflight = 0, inflight_parity = 0;    // thread 0's issued loads
    auto issue = [&](int k) {
        const int item = (int)blockIdx.x + k * (int)gridDim.x;
        if (item >= p.total_items)
            return;
        int d, rb, cc;
        decode_item(p, item, d, rb, cc);
        const int b = k % kBufs;
        const uint32_t bar = bar0 + 8u * b;
        ptx::mbar_arrive_expect_tx(bar, kTileBytes);
        ptx::tma_load_2d(ptx::smem_addr(&tile[b][0]), &p.tm[d], cc * kChunkScales, rb * 128, bar, pol);
        inflight |= 1u << b;
        inflight_parity = (inflight_parity & ~(1u << b)) | ((uint32_t)((k / kBufs) & 1) << b);
    };
    if (threadIdx.x == 0)
        for (int k = 0; k < kBufs; ++k)
            issue(k);

    for (int k = 0;; ++k) {
        const int item = (int)blockIdx.x + k * (int)gridDim.x;
        if (item >= p.total_items)
            break;
        const int b = k % kBufs;
        if (threadIdx.x == 0) {
            // bounded wait for the tile; on expiry record it and stop (uniformly)
            const uint32_t bar = bar0 + 8u * b, par = (uint32_t)((k / kBufs) & 1);
            const uint64_t t0 = ptx::globaltimer_ns();
            int ok = 1;
            while (!ptx::mbar_try_wait(bar, par)) {
                if (ptx::globaltimer_ns() - t0 > p.timeout_ns) {
                    atomicOr(p.err, 1u);
                    ok = 0;
                    break;
                }
            }
            if (ok)
                inflight &= ~(1u << b);
            ok_flag = ok;
        }
        __syncthreads();
        if (!ok_flag)
            break;
        int d, rb, cc;
        decode_item(p, item, d, rb, cc);
        const int kcols = p.kcols[d];
        const int natoms = min(16, (kcols - cc * kChunkScales) / 4);
        const uint8_t *t = tile[b];
        uint8_t *out = p.dst[d] + ((size_t)rb * (kcols / 4) + (size_t)cc * 16) * 512;
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const int idx = threadIdx.x + kThreads * pass;     // 0..511
            const int a = idx & 15;                            // atom
            const int l = 2 * (idx >> 5) + ((idx >> 4) & 1);   // 16-byte row of the atom
            if (a < natoms) {
                uint4 y;
                y.x = *reinterpret_cast<const uint32_t *>(t + (l)*kChunkScales + 4 * a);
                y.y = *reinterpret_cast<const uint32_t *>(t + (l + 32) * kChunkScales + 4 * a);
                y.z = *reinterpret_cast<const uint32_t *>(t + (l + 64) * kChunkScales + 4 * a);
                y.w = *reinterpret_cast<const uint32_t *>(t + (l + 96) * kChunkScales + 4 * a);
                *reinterpret_cast<uint4 *>(out + (size_t)a * 512 + l * 16) = y;
            }
        }
        __syncthreads();    // tile[b] fully read before it is reloaded
        if (threadIdx.x == 0)
            issue(k + kBufs);
    }
    // loads issued but not consumed (after an expired wait) still write this
    // CTA's shared memory: wait for them (bounded) before exiting
    if (threadIdx.x == 0) {
        for (int b = 0; b < kBufs; ++b) {
            if (!(inflight & (1u << b)))
                continue;
            const uint64_t t0 = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(bar0 + 8u * b, (inflight_parity >> b) & 1u))
                if (ptx::globaltimer_ns() - t0 > p.timeout_ns) {
                    atomicOr(p.err, 2u);
                    break;
                }
        }
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

    static thread_local RelayoutParams P;
    auto launch = [&]() -> int {
        if (P.count == 0)
            return NVFP4_OK;
        P.total_items = P.item_end[P.count - 1];
        P.err = dev->err;
        P.timeout_ns = wait_timeout_ns();
        const int max_ctas = dev->sm_count * kCtasPerSm;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(P.total_items < max_ctas ? P.total_items : max_ctas);
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
        const long long n = (long long)rblocks * chunks;
        if (P.count == kMaxDescs || (long long)items + n > (1ll << 30)) {
            rc = launch();
            if (rc != NVFP4_OK)
                return rc;
            P.count = 0;
            items = 0;
        }
        const int j = P.count;
        rc = encode_map_2d(&P.tm[j], CU_TENSOR_MAP_DATA_TYPE_UINT8, d.src, (uint64_t)kcols,
                           (uint64_t)d.rows, (uint64_t)kcols, kChunkScales, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (rc != NVFP4_OK)
            return rc;
        P.count = j + 1;
        P.dst[j] = static_cast<uint8_t *>(d.dst);
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
