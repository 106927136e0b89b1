// runtime.h -- host-side state shared by the library's translation units:
// per-device capability check and set-up, the device error word, the
// tensor-map encoder and the wait-timeout knob.
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>
#include <cstdint>

namespace nvfp4 {

struct DeviceState {
    int initialised;
    int supported;    // compute capability 10.3
    int sm_count;
    uint32_t *err;    // two device words: error bits, first expiry (block << 4 | role)
};

// State of the current device, set up on first use (capability query,
// 16-byte error word, kernel attributes).  Returns an NVFP4_* code.
int current_device(DeviceState **out);

// cuTensorMapEncodeTiled through the runtime's driver entry point, with a
// cache keyed on every argument that varies.  2-D, 128-byte swizzle, 256-byte
// L2 promotion, zero fill out of bounds.  Returns an NVFP4_* code.
int encode_map_2d(CUtensorMap *out, CUtensorMapDataType dtype, const void *ptr, uint64_t dim0,
                  uint64_t dim1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1);

unsigned long long wait_timeout_ns();
int debug_drop_stage();
int b_policy_override();   // -1 = use the built-in choice

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace nvfp4
