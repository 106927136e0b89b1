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
// cache keyed on every argument that varies.  2-D, 256-byte L2 promotion,
// zero fill out of bounds.  Returns an NVFP4_* code.
int encode_map_2d(CUtensorMap *out, CUtensorMapDataType dtype, const void *ptr, uint64_t dim0,
                  uint64_t dim1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1,
                  CUtensorMapSwizzle swizzle);

// K-major packed FP4 operand [rows][K/2] bytes as a 3-D uint8 tensor
// {128 B, rows, K/256} (strides K/2 and 128 bytes), box {128, box_rows,
// box_chunks}, 128-byte swizzle: one load brings box_chunks consecutive
// 128-byte pieces of every row.
int encode_map_operand(CUtensorMap *out, const void *ptr, uint64_t rows, uint64_t K,
                       uint32_t box_rows, uint32_t box_chunks);

// Tiled scale factors of a [rows][K] operand (ceil(rows/128) row blocks of
// K/64 atoms of 512 bytes) as a 3-D uint32 tensor {128, K/64, row blocks},
// box {128, box_atoms, box_blocks}, no swizzle: one load brings the atoms of
// one stage (box_atoms = stage K / 64) for box_blocks consecutive row blocks
// (zeros past the last atom or row block).
int encode_map_sf(CUtensorMap *out, const void *ptr, uint64_t rows, uint64_t K, uint32_t box_atoms,
                  uint32_t box_blocks);
// 16-bit C [rows][cols] (cols a multiple of 64) seen as 64-column blocks:
// {64, rows, cols / 64} with strides {2 cols, 128} bytes, box {64, 32,
// box_blocks}, 128-byte swizzle (one tile's 32-row slab per store)
int encode_map_c_wide(CUtensorMap *out, CUtensorMapDataType dtype, const void *ptr, uint64_t rows,
                      uint64_t cols, uint32_t box_blocks);

// Stream-K scratch of one (device, stream): `slots` partial-sum slots of
// 128 x 256 FP32, four flag words per slot (set to all ones at allocation)
// and the launch epoch with its finished-CTA count (both zero).  Allocated on
// the first request for the pair, never while the stream is capturing a
// graph; kept until the process exits.  Returns an NVFP4_* code.
struct SkScratch {
    float *ws;
    uint32_t *flags;
    uint32_t *epoch;
    int slots;
};
int sk_scratch(cudaStream_t stream, int slots, SkScratch *out);

unsigned long long wait_timeout_ns();
int debug_drop_stage();
int b_policy_override();   // -1 = use the built-in choice
// tuning and debug knobs from the environment, read at every call:
// NVFP4_GEMM_KIND (0 stream, 1 wide, 2 compute, 3 wide with 512-K stages,
// 4 / 5 wide with 2 / 4 producer pairs, 6 CTA pairs),
// NVFP4_PF_STAGES, NVFP4_B_POLICY (0 normal, 1 evict_first, 2 evict_last)
int env_int(const char *name, int fallback);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace nvfp4
