// runtime.cu -- per-device set-up, tensor-map cache, error word, C-ABI
// utility entry points (nvfp4_last_device_error, nvfp4_strerror, ...).
#include "runtime.h"

#include <cudaTypedefs.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <unordered_map>
#include <utility>

#include "../../include/nvfp4_group_gemm.h"

namespace nvfp4 {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
DeviceState g_dev[kMaxDevices];

std::mutex g_map_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
std::atomic<int> g_debug_drop{0};

struct MapKey {
    const void *ptr;
    uint64_t dim0, dim1, dim2, stride1, stride2;
    uint32_t box0, box1, box2;
    int rank, dtype, swizzle;
    bool operator==(const MapKey &o) const
    {
        return ptr == o.ptr && dim0 == o.dim0 && dim1 == o.dim1 && dim2 == o.dim2 &&
               stride1 == o.stride1 && stride2 == o.stride2 && box0 == o.box0 && box1 == o.box1 &&
               box2 == o.box2 && rank == o.rank && dtype == o.dtype && swizzle == o.swizzle;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey &k) const
    {
        uint64_t h = reinterpret_cast<uintptr_t>(k.ptr);
        auto mix = [&](uint64_t v) {
            h ^= v + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
        };
        mix(k.dim0);
        mix(k.dim1);
        mix(k.dim2);
        mix(k.stride1);
        mix(k.stride2);
        mix((uint64_t)k.box0 << 32 | k.box1);
        mix((uint64_t)k.box2 << 32 | (uint64_t)k.rank << 16 | (uint64_t)k.dtype << 8 |
            (uint64_t)k.swizzle);
        return (size_t)h;
    }
};
// one cache per device would be stricter; a tensor map holds only the
// address and shape, which are device-independent values
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;
constexpr size_t kMaxCachedMaps = 8192;

int load_encoder()
{
    if (g_encode)
        return NVFP4_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return NVFP4_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return NVFP4_OK;
}

int read_env_int(const char *name, int fallback)
{
    const char *v = std::getenv(name);
    return v ? std::atoi(v) : fallback;
}

}  // namespace

int current_device(DeviceState **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return NVFP4_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceState &d = g_dev[dev];
    if (!d.initialised) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        d.supported = (major == 10 && minor == 3);
        d.sm_count = sms;
        if (d.supported) {
            void *e = nullptr;
            if (cudaMalloc(&e, 16) != cudaSuccess)
                return NVFP4_ERR_CUDA;
            if (cudaMemset(e, 0, 16) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
                cudaFree(e);
                return NVFP4_ERR_CUDA;
            }
            d.err = static_cast<uint32_t *>(e);
        }
        d.initialised = 1;
    }
    *out = &d;
    return d.supported ? NVFP4_OK : NVFP4_ERR_UNSUPPORTED;
}

namespace {

int encode_map(CUtensorMap *out, const MapKey &key)
{
    std::lock_guard<std::mutex> lk(g_map_mu);
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
        *out = it->second;
        return NVFP4_OK;
    }
    int rc = load_encoder();
    if (rc != NVFP4_OK)
        return rc;
    const cuuint64_t dims[3] = {key.dim0, key.dim1, key.dim2};
    const cuuint64_t strides[2] = {key.stride1, key.stride2};
    const cuuint32_t box[3] = {key.box0, key.box1, key.box2};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(out, (CUtensorMapDataType)key.dtype, (cuuint32_t)key.rank,
                          const_cast<void *>(key.ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, (CUtensorMapSwizzle)key.swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return NVFP4_ERR_INVALID_ARGUMENT;
    if (g_maps.size() >= kMaxCachedMaps)
        g_maps.clear();
    g_maps.emplace(key, *out);
    return NVFP4_OK;
}

}  // namespace

int encode_map_2d(CUtensorMap *out, CUtensorMapDataType dtype, const void *ptr, uint64_t dim0,
                  uint64_t dim1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1,
                  CUtensorMapSwizzle swizzle)
{
    const MapKey key{ptr, dim0, dim1, 1, stride1_bytes, 0, box0, box1, 1, 2, (int)dtype, (int)swizzle};
    return encode_map(out, key);
}

int encode_map_operand(CUtensorMap *out, const void *ptr, uint64_t rows, uint64_t K,
                       uint32_t box_rows, uint32_t box_chunks)
{
    const MapKey key{ptr,   128, rows,     K / 256,    K / 2, 128, 128, box_rows, box_chunks, 3,
                     (int)CU_TENSOR_MAP_DATA_TYPE_UINT8, (int)CU_TENSOR_MAP_SWIZZLE_128B};
    return encode_map(out, key);
}

int encode_map_sf(CUtensorMap *out, const void *ptr, uint64_t rows, uint64_t K, uint32_t box_atoms,
                  uint32_t box_blocks)
{
    const uint64_t atoms = K / 64;
    const MapKey key{ptr, 128, atoms, (rows + 127) / 128, 512, atoms * 512, 128, box_atoms, box_blocks, 3,
                     (int)CU_TENSOR_MAP_DATA_TYPE_UINT32, (int)CU_TENSOR_MAP_SWIZZLE_NONE};
    return encode_map(out, key);
}

int encode_map_c_wide(CUtensorMap *out, CUtensorMapDataType dtype, const void *ptr, uint64_t rows,
                      uint64_t cols, uint32_t box_blocks)
{
    const MapKey key{ptr, 64, rows, cols / 64, cols * 2, 128, 64, 32, box_blocks, 3, (int)dtype,
                     (int)CU_TENSOR_MAP_SWIZZLE_128B};
    return encode_map(out, key);
}

namespace {
std::mutex g_sk_mu;
std::map<std::pair<int, cudaStream_t>, SkScratch> g_sk;
}  // namespace

int sk_scratch(cudaStream_t stream, int slots, SkScratch *out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_sk_mu);
    auto it = g_sk.find({dev, stream});
    if (it != g_sk.end() && it->second.slots >= slots) {
        *out = it->second;
        return NVFP4_OK;
    }
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
        return NVFP4_ERR_UNSUPPORTED;
    const size_t ws_bytes = (size_t)slots * 128 * 256 * sizeof(float);
    const size_t flag_bytes = (size_t)slots * 4 * sizeof(uint32_t);
    void *mem = nullptr;
    if (cudaMalloc(&mem, ws_bytes + flag_bytes + 16) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    SkScratch s;
    s.ws = static_cast<float *>(mem);
    s.flags = reinterpret_cast<uint32_t *>(static_cast<char *>(mem) + ws_bytes);
    s.epoch = reinterpret_cast<uint32_t *>(static_cast<char *>(mem) + ws_bytes + flag_bytes);
    s.slots = slots;
    // flags all ones, epoch 0: no flag matches before a partial is written
    if (cudaMemsetAsync(s.flags, 0xFF, flag_bytes, stream) != cudaSuccess ||
        cudaMemsetAsync(s.epoch, 0, 16, stream) != cudaSuccess) {
        cudaFree(mem);
        return NVFP4_ERR_CUDA;
    }
    // a smaller area of this stream is left in place: launches already
    // queued on the stream may still use it
    g_sk[{dev, stream}] = s;
    *out = s;
    return NVFP4_OK;
}

unsigned long long wait_timeout_ns() { return g_timeout_ns.load(std::memory_order_relaxed); }
int debug_drop_stage() { return g_debug_drop.load(std::memory_order_relaxed); }
int b_policy_override() { return read_env_int("NVFP4_B_POLICY", -1); }
int env_int(const char *name, int fallback) { return read_env_int(name, fallback); }

}  // namespace nvfp4

extern "C" {

int nvfp4_last_device_error(cudaStream_t stream)
{
    if (cudaStreamSynchronize(stream) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    nvfp4::DeviceState *d = nullptr;
    int rc = nvfp4::current_device(&d);
    if (rc != NVFP4_OK)
        return rc;
    uint32_t h[2] = {0, 0};
    if (cudaMemcpy(h, d->err, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (h[0] == 0)
        return NVFP4_OK;
    if (cudaMemset(d->err, 0, sizeof(h)) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    return NVFP4_ERR_TIMEOUT;
}

void nvfp4_set_wait_timeout_ns(uint64_t ns)
{
    if (ns < 1000000ull)
        ns = 1000000ull;
    nvfp4::g_timeout_ns.store(ns, std::memory_order_relaxed);
}

void nvfp4_debug_drop_first_stage(int enable)
{
    nvfp4::g_debug_drop.store(enable ? 1 : 0, std::memory_order_relaxed);
}

const char *nvfp4_strerror(int code)
{
    switch (code) {
    case NVFP4_OK:
        return "success";
    case NVFP4_ERR_INVALID_ARGUMENT:
        return "invalid argument";
    case NVFP4_ERR_MISALIGNED:
        return "pointer not 16-byte aligned";
    case NVFP4_ERR_UNSUPPORTED:
        return "current device is not compute capability 10.3 (sm_103a)";
    case NVFP4_ERR_CUDA:
        return "CUDA runtime or driver error";
    case NVFP4_ERR_TIMEOUT:
        return "a bounded wait inside a kernel expired";
    case NVFP4_ERR_TOO_MANY:
        return "size exceeds a documented limit";
    default:
        return "unknown error code";
    }
}

int nvfp4_version(void) { return (0 << 16) | (1 << 8) | 0; }

}  // extern "C"
