// quantize.cu -- NVFP4 quantisation kernel and its C-ABI entry point
// (nvfp4_quantize): FP16 / BF16 [rows][K] -> the grouped GEMM's operand
// format, E2M1 codes [rows][K/2] plus E4M3FN scales per 16 elements, the
// scales written directly in the tiled layout the GEMM reads (and, when
// asked, also row-major).
//
// Per 16-element block of a row (the generator of the "quantized" grouped
// GEMM configuration: values quantised per 16-block to E2M1 with an
// absmax/6 scale rounded to E4M3FN):
//   s    = E4M3FN(absmax / 6)        round to nearest even, saturating at 448
//   code = E2M1(x / decode(s))        round to nearest even, saturating at 6
// both taken on IEEE single-precision values (the quotients rounded to
// nearest); a zero magnitude is stored as code 0 (no sign), and a block whose
// scale rounds to 0 gets codes 0.  The conversions are the hardware's
// cvt.rn.satfinite to e4m3x2 / e2m1x2.
//
// One CTA of 128 threads takes one 128-row block and one 64-element K block
// (one 512-byte scale atom): thread t reads row t's 128 bytes of input, writes
// its 32 bytes of codes, and its four scales into the atom staged in shared
// memory; one warp then stores the atom with 16-byte stores.  Algorithmic
// traffic: 2 bytes read and 0.5 + 1/16 (+ 1/16 row-major) bytes written per
// element; the exact single-precision division per element makes it about
// 20 instructions per element, so issue and memory latency share the bound.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "../../include/nvfp4_group_gemm.h"
#include "ptx.cuh"
#include "runtime.h"

namespace nvfp4 {
namespace {

constexpr int kMaxDim = 1 << 20;
constexpr int kRows = 128;       // rows per CTA (one scale row block)
constexpr int kColsPerCta = 64;  // K elements per CTA (one scale atom)

__device__ __forceinline__ uint32_t e4m3_of(float s)
{
    uint32_t e;
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\tcvt.u32.u16 %0, t;\n\t}"
        : "=r"(e)
        : "f"(0.0f), "f"(s));
    return e & 0xFFu;
}

__device__ __forceinline__ float e4m3_value(uint32_t e)
{
    uint32_t h;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h) : "r"(e));
    return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

// E2M1 codes of (lo, hi), lo in bits 0..3; a zero magnitude loses its sign
__device__ __forceinline__ uint32_t e2m1x2_of(float lo, float hi)
{
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tmov.b32 %0, {t, 0, 0, 0};\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    r &= 0xFFu;
    if ((r & 0x7u) == 0)
        r &= 0xF0u;
    if ((r & 0x70u) == 0)
        r &= 0x0Fu;
    return r;
}

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (BF16) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        } else {
            f[2 * i] = __half2float(__ushort_as_half((unsigned short)(w[i] & 0xFFFFu)));
            f[2 * i + 1] = __half2float(__ushort_as_half((unsigned short)(w[i] >> 16)));
        }
    }
}

struct QuantParams {
    const uint16_t *x;
    uint8_t *codes;
    uint8_t *sf_tiled;
    uint8_t *sf_rowmajor;   // may be null
    int rows, K;
};

// One CTA: 128 rows x 64 elements (one scale atom); thread t takes row t:
// eight 16-byte loads (its whole 128-byte row segment, issued before the
// first use), four 16-element blocks, 32 bytes of codes in two 16-byte
// stores, and its four scales into the atom staged in shared memory.
template <bool BF16>
__global__ void __launch_bounds__(kRows) quantize_kernel(const __grid_constant__ QuantParams p)
{
    __shared__ __align__(16) uint32_t atom[kRows];   // 512 bytes
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();

    const int kb = blockIdx.x;                  // 64-element K block
    const int rb = blockIdx.y;                  // 128-row block
    const int t = threadIdx.x;
    const int r = rb * kRows + t;
    uint32_t sfw = 0;                           // the row's four scales
    if (r < p.rows) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.x + (size_t)r * p.K + (size_t)kb * kColsPerCta);
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = __ldg(src + i);
        uint32_t cw[8];                         // 32 bytes of codes
#pragma unroll
        for (int j = 0; j < 4; ++j) {           // 16-element blocks
            float lo8[8], hi8[8];
            unpack8<BF16>(v[2 * j], lo8);
            unpack8<BF16>(v[2 * j + 1], hi8);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                amax = fmaxf(amax, fmaxf(fabsf(lo8[i]), fabsf(hi8[i])));
            const uint32_t sc = e4m3_of(amax / 6.0f);
            const float sdec = e4m3_value(sc);
            sfw |= sc << (8 * j);
            uint32_t b[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                b[i] = sdec > 0.0f ? e2m1x2_of(lo8[2 * i] / sdec, lo8[2 * i + 1] / sdec) : 0u;
                b[4 + i] = sdec > 0.0f ? e2m1x2_of(hi8[2 * i] / sdec, hi8[2 * i + 1] / sdec) : 0u;
            }
            cw[2 * j] = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
            cw[2 * j + 1] = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(p.codes + (size_t)r * (p.K / 2) + (size_t)kb * (kColsPerCta / 2));
        dst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
        dst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
        if (p.sf_rowmajor)
            *reinterpret_cast<uint32_t *>(p.sf_rowmajor + (size_t)r * (p.K / 16) + (size_t)kb * 4) = sfw;
    }
    // row t's four scales at byte (t % 32) * 16 + (t / 32) * 4 of the atom;
    // rows past `rows` stay zero
    atom[(t % 32) * 4 + t / 32] = sfw;
    __syncthreads();
    if (t < 32) {
        const uint4 w = reinterpret_cast<const uint4 *>(atom)[t];
        uint4 *dst = reinterpret_cast<uint4 *>(p.sf_tiled + ((size_t)rb * (p.K / 64) + kb) * 512);
        dst[t] = w;
    }
}

}  // namespace
}  // namespace nvfp4

extern "C" int nvfp4_quantize(const void *x, int x_is_bf16, int rows, int K, void *codes, void *sf_tiled,
                              void *sf_rowmajor, cudaStream_t stream)
{
    using namespace nvfp4;
    if (rows < 0 || K <= 0 || K % kColsPerCta != 0 || rows > kMaxDim || K > kMaxDim)
        return NVFP4_ERR_INVALID_ARGUMENT;
    if (rows == 0)
        return NVFP4_OK;
    if (!x || !codes || !sf_tiled)
        return NVFP4_ERR_INVALID_ARGUMENT;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(sf_tiled) || (sf_rowmajor && !aligned16(sf_rowmajor)))
        return NVFP4_ERR_MISALIGNED;
    DeviceState *dev = nullptr;
    int rc = current_device(&dev);
    if (rc != NVFP4_OK)
        return rc;
    QuantParams p;
    p.x = static_cast<const uint16_t *>(x);
    p.codes = static_cast<uint8_t *>(codes);
    p.sf_tiled = static_cast<uint8_t *>(sf_tiled);
    p.sf_rowmajor = static_cast<uint8_t *>(sf_rowmajor);
    p.rows = rows;
    p.K = K;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(K / kColsPerCta, (rows + kRows - 1) / kRows);
    cfg.blockDim = dim3(kRows);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = env_int("NVFP4_PDL", 1) != 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = x_is_bf16 ? cudaLaunchKernelEx(&cfg, quantize_kernel<true>, p)
                                    : cudaLaunchKernelEx(&cfg, quantize_kernel<false>, p);
    if (e != cudaSuccess || cudaGetLastError() != cudaSuccess)
        return NVFP4_ERR_CUDA;
    return NVFP4_OK;
}
