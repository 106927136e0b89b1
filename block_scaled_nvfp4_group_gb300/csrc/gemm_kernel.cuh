// gemm_kernel.cuh -- persistent, warp-specialised NVFP4 grouped GEMM for
// sm_103a (GB300).
//
// One CTA per SM walks a flat list of output tiles of every group
// (tile t, t + gridDim.x, ...).  Warps and roles:
//   warps 0-3  epilogue: tensor memory -> registers (tcgen05.ld), FP32 ->
//              FP16 (round to nearest even), a swizzled shared-memory tile
//              per warp and a TMA tensor store, which writes whole row
//              segments and clips rows >= M and columns >= N;
//   warps 6-9  loaders, one TMA thread each, one operation per stage each:
//              the A tile [128 x BK/2 bytes] and the B tile [BN x BK/2 bytes]
//              (3-D boxes over 128-byte K chunks, 128-byte swizzle) complete
//              on full[slot]; the A and B scale atoms of the stage (3-D boxes
//              over the tiled scales) complete on sf_full[slot].  A thread
//              issues only a few TMA operations per microsecond on GB300, so
//              the stage's operations are spread over four threads;
//   warp 10    L2 prefetcher (optional): B tiles and scales of the stages up
//              to `pf_stages` ahead of the MMAs, beyond what the ring holds;
//   warp 5     scale copier (one thread): once a stage's scales have landed
//              (sf_full, ahead of the larger operand tiles), tcgen05.cp of its
//              atoms into the slot's own tensor-memory columns, then
//              tcgen05.commit to sf_ready[slot];
//   warp 4     MMA issuer (one thread): after full[slot] and sf_ready[slot],
//              BK/64 tcgen05.mma.kind::mxf4nvf4.block_scale.block16
//              (128 x BN x 64) per stage into an FP32 accumulator (two of them
//              when BN=128), and tcgen05.commit to free the stage / hand the
//              accumulator on.
// The epilogue hands the accumulator back as soon as it holds the tile in
// registers (as FP16), so its stores overlap the MMAs of the next tile; with
// two accumulators (BN = 128) the MMAs do not even wait for its loads.
//
// The warp roles, the scale addressing and the descriptor fields follow
// kernelbot nvfp4-group-gemm submission 474067 (group_gemm_persistent_kernel,
// tcgen05_mma_nvfp4, tcgen05_cp_nvfp4, the TMA producer warp); the split
// loaders, the separate scale barrier, the store path, the bounded waits and
// the tensor-memory budget are not taken from that page.
//
// Every mbarrier wait is bounded: when it expires the waiting role sets the
// device error word and a shared abort flag, all roles leave their loops, the
// loaders wait (bounded) for the copies they issued, the MMA thread waits
// for its issued tensor-core work, the epilogue waits for its stores, and the
// CTA frees its tensor memory and exits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"

namespace nvfp4 {

constexpr int kBM = 128;           // MMA M, rows of A per tile
constexpr int kChunkK = 256;       // K elements per 128-byte chunk of a row
constexpr int kMmaK = 64;          // K elements per tcgen05.mma (FP4)
constexpr int kMaxGroups = 32;     // groups per launch (param block)
constexpr int kMmaWarp = 4;        // MMA issuer; also allocates / frees tensor memory
constexpr int kSfWarp = 5;         // scale copies shared -> tensor memory
constexpr int kFirstLoaderWarp = 6;  // A, B, A scales, B scales
constexpr int kLoaderRoles = 4;
constexpr int kSmemLimit = 232448; // 227 KiB per CTA

// error word bits (device_err[0]); device_err[1] records who expired first
constexpr uint32_t kErrTimeout = 1u;
constexpr uint32_t kErrDrainTimeout = 2u;

enum : uint32_t {
    kRoleProducer = 1,
    kRoleMma = 2,
    kRoleEpilogue = 3,
    kRoleDrain = 4,
    kRoleSf = 5,
    kRoleStreamK = 6   // an epilogue warp waiting for another CTA's partial sum
};

struct GemmParams {
    CUtensorMap tmA[kMaxGroups];  // uint8 {128 B, M, K/256}, box {128, 128, BK/256}, 128B swizzle
    CUtensorMap tmB[kMaxGroups];  // uint8 {128 B, N, K/256}, box {128, BN, BK/256}
    CUtensorMap tmC[kMaxGroups];  // fp16 [M][N], box EPI_COLS x 32, swizzle = EPI_COLS * 2 B
    // C as 64-column blocks, {64, M, N/64} with strides {2N, 128} bytes, box
    // {64, 32, tile columns / 64}, 128-byte swizzle: the whole 32-row slab of
    // a tile in one store (used for a CTA's last tile; c_wide[g] = 0 when N
    // is not a multiple of 64)
    CUtensorMap tmCw[kMaxGroups];
    int c_wide[kMaxGroups];
    int M[kMaxGroups];
    int N[kMaxGroups];
    int kchunks[kMaxGroups];   // K / 256
    int grid_m[kMaxGroups];    // ceil(M / 128)
    int tile_end[kMaxGroups];  // inclusive prefix sum of grid_m * grid_n
    int num_groups;
    int total_tiles;
    uint32_t *err;             // device error words [2]
    unsigned long long timeout_ns;
    int b_policy;              // L2 policy of B / SFB loads: 0 normal, 1 first, 2 last
    int pf_stages;             // L2 prefetch distance for B, in stages ahead of the ring (0 = off)
    int debug_drop_stage;      // test hook: CTA 0's B loader never issues its first stage
    // fused epilogue: C = alpha[g] * A B^T (or its SwiGLU), FP16 or BF16
    float alpha[kMaxGroups];
    int out_bf16;              // C elements: 0 FP16, 1 BF16
    int swiglu;                // 1: every 256-column tile = 128 gate + 128 up columns, C is [M][N/2]
    // 1: A and B were complete before the kernel preceding this launch in
    // the stream began (the library's own relayout + GEMM call), so their
    // loads need not wait for that kernel to finish
    int early_ab;
    // stream-K launches: the flat sequence of (tile, k-stage) units, tiles in
    // list order, is cut into gridDim.x contiguous ranges, CTA c taking units
    // [c U / G, (c + 1) U / G) with U = units_total
    int units_total;
    int unit_end[kMaxGroups];  // inclusive prefix sum of tiles x stages
    float *sk_ws;              // per CTA one partial accumulator, 128 x BN FP32
    uint32_t *sk_flags;        // per CTA and epilogue warp: epoch of its last partial
    uint32_t *sk_epoch;        // [0] epoch of the launch, [1] CTAs finished
};

// Parameter block of a launch: the GEMM parameters and the 3-D maps of the
// tiled scales (uint32 {128, K/64, row blocks}: one 512-byte atom per
// (row block, 64-K block)), whose box covers the atoms of one stage for the
// row blocks of one tile.
struct KernelParams {
    GemmParams g;
    CUtensorMap tmSFA[kMaxGroups];  // box {128, BK/64, 1}
    CUtensorMap tmSFB[kMaxGroups];  // box {128, BK/64, BN/128} (BN/2 per CTA of a pair: 128 rows each)
};
static_assert(sizeof(KernelParams) <= 32764, "kernel parameter block over 32 KiB");

// BN: tile width; BK: K elements per stage (256 or 512); STAGES: ring depth;
// EPI_COLS: columns per epilogue store (32 or 64); EPI_BUFS: staging
// buffers per epilogue warp (1 or 2)
template <int BN_, int BK_, int STAGES_, int EPI_COLS_, int EPI_BUFS_>
struct GemmConfig {
    static constexpr int BN = BN_;
    static constexpr int BK = BK_;
    static constexpr int kStages = STAGES_;
    static constexpr int kPrefetchWarp = kFirstLoaderWarp + kLoaderRoles;
    static constexpr int kThreads = 32 * (kPrefetchWarp + 1);
    static_assert(kThreads <= 1024, "too many warps");
    static constexpr int kEpiCols = EPI_COLS_;
    static constexpr int kEpiBufs = EPI_BUFS_;
    static_assert(BN == 128 || BN == 256, "BN must be 128 or 256");
    static_assert(BK == 256 || BK == 512, "BK must be 256 or 512");
    static_assert(kEpiCols == 32 || kEpiCols == 64, "epilogue chunk must be 32 or 64 columns");
    static_assert(kEpiBufs == 1 || kEpiBufs == 2, "one or two staging buffers per warp");
    static constexpr int kChunks = BK / kChunkK;           // 128-byte chunks per row per stage
    static constexpr int kMmas = BK / kMmaK;               // MMAs per stage (4 or 8)
    static constexpr int kAccBufs = (BN == 128) ? 2 : 1;
    static constexpr int kABytes = kBM * BK / 2;
    static constexpr int kBBytes = BN * BK / 2;
    static constexpr int kSfaBytes = kMmas * 512;          // one atom per 64 K
    static constexpr int kSfbBytes = (BN / 128) * kMmas * 512;
    static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1 KiB alignment");
    static constexpr int kEpiBufBytes = 32 * kEpiCols * 2;  // 32 rows of one chunk
    static constexpr int kEpiOff = kStages * kStageBytes;
    static constexpr int kBarOff = kEpiOff + 4 * kEpiBufs * kEpiBufBytes;
    // full[S], empty[S], sf_ready[S], sf_full[S], acc_full[2], acc_empty[2],
    // drain, sf_drain
    static constexpr int kNumBars = 4 * kStages + 6;
    static constexpr int kSlotOff = kBarOff + 8 * kNumBars;  // tmem base, abort flag, MMA progress
    static constexpr int kSmemBytes = kSlotOff + 16 + 1024;  // + alignment slack
    static_assert(kSmemBytes <= kSmemLimit, "exceeds 227 KiB of shared memory");
    static_assert(kStages * kStageBytes >= 4 * (BN / 64) * 4096, "ring too small for the last tile's slabs");
    // tensor memory: accumulators, then one scale region per ring slot
    // (SFA atoms, then SFB atoms): the copies for stage q+1 never write the
    // columns the MMAs of stage q read, so they need not wait for them
    static constexpr int kTmemCols = 512;
    static constexpr int kSfCol0 = kAccBufs * BN;
    static constexpr int kSfSlotCols = 4 * kMmas * (1 + BN / 128);
    static_assert(kSfCol0 + kStages * kSfSlotCols <= kTmemCols, "tensor memory budget");
    static constexpr uint32_t sfa_col(int slot, int j) { return kSfCol0 + slot * kSfSlotCols + 4 * j; }
    static constexpr uint32_t sfb_col(int slot, int j, int h)
    {
        return kSfCol0 + slot * kSfSlotCols + 4 * kMmas + 4 * (BN / 128) * j + 4 * h;
    }
    // instruction descriptor (kind::mxf4nvf4): A and B E2M1 (format 1) at
    // bits 7 and 10, both K-major, N>>3 at bit 17, UE4M3 scales (bit 23 = 0),
    // M>>7 at bit 27, scale-factor data ids 0
    static constexpr uint32_t kIdesc =
        (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kBM >> 7) << 27);
};

// shared-memory matrix descriptor, K-major operand tile with 128-byte
// swizzle: 8-row groups 1024 bytes apart, descriptor version 1 (bit 46)
__device__ __forceinline__ uint64_t desc_operand_sw128(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}

// descriptor of one 512-byte scale atom (32 rows x 16 bytes, no swizzle,
// 8-row groups 128 bytes apart)
__device__ __forceinline__ uint64_t desc_scale_atom(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 32) | (1ull << 46);
}

struct TileCoord {
    int g, bm, bn;
};

// advance the running group index to the group holding tile t (t only grows
// within one CTA) and split the group-local index, M-tile fastest, so that
// the M-tiles sharing one B strip are neighbours in the list
__device__ __forceinline__ TileCoord tile_coord(const GemmParams &p, int t, int &g)
{
    while (t >= p.tile_end[g])
        ++g;
    int local = t - (g > 0 ? p.tile_end[g - 1] : 0);
    int gm = p.grid_m[g];
    return TileCoord{g, local % gm, local / gm};
}

struct WaitCtx {
    volatile uint32_t *abort;
    uint32_t *err;
    unsigned long long timeout_ns;
};

__device__ __noinline__ bool wait_bounded_slow(uint32_t bar, uint32_t parity, const WaitCtx &w,
                                               uint32_t role)
{
    const uint64_t t0 = ptx::globaltimer_ns();
    for (;;) {
        if (ptx::mbar_try_wait(bar, parity))
            return true;
        if (*w.abort)
            return false;
        if (ptx::globaltimer_ns() - t0 > w.timeout_ns) {
            *w.abort = 1u;
            atomicOr(w.err, kErrTimeout);
            atomicCAS(w.err + 1, 0u, (blockIdx.x << 4) | role);
            return false;
        }
    }
}

// bounded wait: true once the phase completed; false when another role
// aborted or when this wait expired (then the error word and abort flag are
// set)
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtx &w,
                                             uint32_t role)
{
    if (ptx::mbar_try_wait(bar, parity))
        return true;
    return wait_bounded_slow(bar, parity, w, role);
}

// bounded wait used while draining after an abort (ignores the abort flag)
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity, const WaitCtx &w)
{
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > w.timeout_ns) {
            atomicOr(w.err, kErrDrainTimeout);
            atomicCAS(w.err + 1, 0u, (blockIdx.x << 4) | kRoleDrain);
            return;
        }
    }
}

// stream-K: bounded wait until another CTA has published `value` in `flag`
// (release / acquire at GPU scope); false when it expired (error word and
// abort flag set) or another role aborted
__device__ __noinline__ bool wait_flag_bounded(const uint32_t *flag, uint32_t value, const WaitCtx &w)
{
    const uint64_t t0 = ptx::globaltimer_ns();
    for (;;) {
        if (ptx::ld_acquire_gpu(flag) == value)
            return true;
        if (*w.abort)
            return false;
        if (ptx::globaltimer_ns() - t0 > w.timeout_ns) {
            *w.abort = 1u;
            atomicOr(w.err, kErrTimeout);
            atomicCAS(w.err + 1, 0u, (blockIdx.x << 4) | kRoleStreamK);
            return false;
        }
        __nanosleep(64);
    }
}

// Stream-K partial accumulators: CTA c's slot holds 128 rows x BN FP32 values
// with element (r, x) in float4 number (x / 4) * 128 + r, so a warp's 32 rows
// of four columns are 512 contiguous bytes on both sides.
template <int BN>
__device__ __forceinline__ void store_partial(float *ws, uint32_t row_taddr, int n0, int N, int row)
{
    float4 *d4 = reinterpret_cast<float4 *>(ws + (size_t)blockIdx.x * (BN * 128)) + row;
#pragma unroll
    for (int c = 0; c < BN / 32; ++c) {
        if (n0 + c * 32 < N) {   // warp-uniform
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(row_taddr + c * 32, v);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i)
                __stcg(d4 + (c * 8 + i) * 128,
                       make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                   __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])));
        }
    }
}

// adds the partial sums of CTAs [h0, h1) to 32 accumulator columns (chunk
// `chunk` of 32) of this thread's row
template <int BN>
__device__ __forceinline__ void add_partials(uint32_t (&v)[32], const float *ws, int h0, int h1, int chunk,
                                             int row)
{
    for (int hc = h0; hc < h1; ++hc) {
        const float4 *s4 = reinterpret_cast<const float4 *>(ws + (size_t)hc * (BN * 128)) + row;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 a = __ldcg(s4 + (chunk * 8 + i) * 128);
            v[4 * i] = __float_as_uint(__uint_as_float(v[4 * i]) + a.x);
            v[4 * i + 1] = __float_as_uint(__uint_as_float(v[4 * i + 1]) + a.y);
            v[4 * i + 2] = __float_as_uint(__uint_as_float(v[4 * i + 2]) + a.z);
            v[4 * i + 3] = __float_as_uint(__uint_as_float(v[4 * i + 3]) + a.w);
        }
    }
}

__device__ __forceinline__ uint32_t pack_out2(float lo, float hi, bool bf16)
{
    if (bf16) {
        __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&b);
    }
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float silu(float x) { return x / (1.0f + __expf(-x)); }

// Epilogue stores of a CTA's last tile (the operand ring is idle): the
// warp's 32 rows x `ocols` output columns as 64-column blocks of 32 rows x
// 128 bytes with the 128-byte swizzle (16-byte chunk q of row r at q ^ (r % 8):
// conflict-free), then a single 3-D tensor store for the warp -- one TMA
// operation instead of one per EC columns.  `buf` is 1024-byte aligned and
// holds BN / 64 blocks of 4 KiB.
template <int BN>
__device__ __forceinline__ void store_slab_wide(const CUtensorMap *tm, uint32_t buf, int lane, int on0, int oN,
                                                int ocols, int m0, const uint32_t (&h)[BN / 2])
{
#pragma unroll
    for (int ch = 0; ch < BN / 64; ++ch) {
        if (ch * 64 < ocols && on0 + ch * 64 < oN) {   // warp-uniform
            const uint32_t row = buf + (uint32_t)ch * 4096u + (uint32_t)lane * 128u;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                ptx::st_shared_v4(row + ((q ^ (lane & 7)) << 4), h[ch * 32 + 4 * q], h[ch * 32 + 4 * q + 1],
                                  h[ch * 32 + 4 * q + 2], h[ch * 32 + 4 * q + 3]);
        }
    }
    ptx::fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
        ptx::tma_store_3d(tm, buf, 0, m0, on0 / 64);
        ptx::bulk_commit_group();
    }
    __syncwarp();
}

// Epilogue, part 1: this thread's accumulator row of the tile (tensor-memory
// lane `row_taddr`, columns [0, BN)) -> packed 16-bit output pairs in
// registers, alpha applied; with SwiGLU, output column c of the tile is
// silu(alpha * acc[c]) * alpha * acc[c + BN/2].  Column chunks at or past N
// (input columns) are skipped.  Every lane of the warp takes part (the
// tensor-memory loads are warp-collective).  With stream-K (SK) the partial
// sums of CTAs [h0, h1) are added to the accumulator first.
template <int BN, bool EPI_EX, bool SK = false>
__device__ __forceinline__ void epilogue_load(const GemmParams &p, int g, uint32_t row_taddr, int n0,
                                              int N, uint32_t (&h)[BN / 2], int h0 = 0, int h1 = 0,
                                              int row = 0)
{
    if constexpr (!EPI_EX) {
        // plain FP16
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
            if (n0 + c * 32 < N) {   // warp-uniform
                uint32_t v[32];
                ptx::tmem_ld_32x32b_x32(row_taddr + c * 32, v);
                ptx::tmem_wait_ld();
                if constexpr (SK)
                    add_partials<BN>(v, p.sk_ws, h0, h1, c, row);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    h[c * 16 + i] = pack_out2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]), false);
            }
        }
        return;
    }
    const float alpha = p.alpha[g];
    const bool bf = p.out_bf16 != 0;
    if (!p.swiglu) {
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
            if (n0 + c * 32 < N) {   // warp-uniform
                uint32_t v[32];
                ptx::tmem_ld_32x32b_x32(row_taddr + c * 32, v);
                ptx::tmem_wait_ld();
                if constexpr (SK)
                    add_partials<BN>(v, p.sk_ws, h0, h1, c, row);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    h[c * 16 + i] = pack_out2(alpha * __uint_as_float(v[2 * i]),
                                              alpha * __uint_as_float(v[2 * i + 1]), bf);
            }
        }
    } else {
#pragma unroll
        for (int c = 0; c < BN / 64; ++c) {     // gate chunk c, up chunk c + BN/64
            uint32_t gv[32], uv[32];
            ptx::tmem_ld_32x32b_x32(row_taddr + c * 32, gv);
            ptx::tmem_ld_32x32b_x32(row_taddr + BN / 2 + c * 32, uv);
            ptx::tmem_wait_ld();
            if constexpr (SK) {
                add_partials<BN>(gv, p.sk_ws, h0, h1, c, row);
                add_partials<BN>(uv, p.sk_ws, h0, h1, c + BN / 64, row);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float o0 = silu(alpha * __uint_as_float(gv[2 * i])) * (alpha * __uint_as_float(uv[2 * i]));
                const float o1 =
                    silu(alpha * __uint_as_float(gv[2 * i + 1])) * (alpha * __uint_as_float(uv[2 * i + 1]));
                h[c * 16 + i] = pack_out2(o0, o1, bf);
            }
        }
    }
}

// stages of a tile: ceil(K / BK); the last one covers only K % BK when K is
// not a multiple of BK (one 256-element chunk of a 512-element stage)
template <int BK>
__device__ __forceinline__ int stages_of(int kchunks)
{
    return (kchunks * kChunkK + BK - 1) / BK;
}

// 64-element K blocks (= scale atoms per row block, = MMAs) of stage `it`
template <int BK>
__device__ __forceinline__ int kblocks_in_stage(int kchunks, int it)
{
    const int left = kchunks * (kChunkK / kMmaK) - it * (BK / kMmaK);
    return left < BK / kMmaK ? left : BK / kMmaK;
}

// A piece of a CTA's work: stages [it0, it1) of the nst stages of tile
// (g, bm, bn).  Whole tiles unless the launch is stream-K, where a tile may
// be cut between CTAs; u1 is then the unit just past the tile's last stage.
struct Piece {
    int g, bm, bn;
    int it0, it1, nst;
    int u1;
};

// first unit of CTA c's stream-K range
__device__ __forceinline__ int sk_begin(const GemmParams &p, int c)
{
    return (int)(((long long)c * p.units_total) / (long long)gridDim.x);
}

// Walks the pieces of one CTA in order: tiles blockIdx.x, + gridDim.x, ...
// whole (SK = false), or the CTA's contiguous range of units (SK = true),
// whose first piece may start and whose last piece may end inside a tile.
// Every role of the CTA walks the same sequence.
template <int BK, bool SK>
struct PieceCursor {
    int g, t, u, e;
    __device__ __forceinline__ void start(const GemmParams &p)
    {
        g = 0;
        if constexpr (SK) {
            u = sk_begin(p, blockIdx.x);
            e = sk_begin(p, blockIdx.x + 1);
        } else {
            t = blockIdx.x;
        }
    }
    __device__ __forceinline__ bool next(const GemmParams &p, Piece &pc)
    {
        if constexpr (!SK) {
            if (t >= p.total_tiles)
                return false;
            const TileCoord tc = tile_coord(p, t, g);
            pc.g = tc.g;
            pc.bm = tc.bm;
            pc.bn = tc.bn;
            pc.nst = stages_of<BK>(p.kchunks[tc.g]);
            pc.it0 = 0;
            pc.it1 = pc.nst;
            pc.u1 = 0;
            t += gridDim.x;
            return true;
        } else {
            if (u >= e)
                return false;
            while (u >= p.unit_end[g])
                ++g;
            const int ub = g > 0 ? p.unit_end[g - 1] : 0;
            const int nst = stages_of<BK>(p.kchunks[g]);
            const int local = u - ub;
            const int lt = local / nst;
            pc.g = g;
            pc.bm = lt % p.grid_m[g];
            pc.bn = lt / p.grid_m[g];
            pc.nst = nst;
            pc.it0 = local - lt * nst;
            pc.it1 = (nst - pc.it0 < e - u) ? nst : pc.it0 + (e - u);
            pc.u1 = ub + (lt + 1) * nst;
            u += pc.it1 - pc.it0;
            return true;
        }
    }
    // after next(): the piece just returned is this CTA's last
    __device__ __forceinline__ bool done(const GemmParams &p) const
    {
        if constexpr (SK)
            return u >= e;
        else
            return t >= p.total_tiles;
    }
};

// One loader role (one thread) of a CTA: ROLE 0 the A tile, 1 the B tile
// (both complete on full[slot]), 2 the A scale atoms, 3 the B scale atoms
// (both on sf_full[slot]).  One arrive.expect_tx and one TMA operation per
// stage; boxes that reach past K or past the rows land as zeros and still
// count their full size.
template <class Cfg, bool SK, int ROLE>
__device__ __forceinline__ void loader_role(const KernelParams &kp, uint32_t base, uint32_t bar0,
                                            const WaitCtx &wctx)
{
    const GemmParams &p = kp.g;
    constexpr int S = Cfg::kStages;
    constexpr bool kSf = ROLE >= 2;
    constexpr uint32_t kOff = ROLE == 0   ? 0u
                              : ROLE == 1 ? (uint32_t)Cfg::kABytes
                              : ROLE == 2 ? (uint32_t)(Cfg::kABytes + Cfg::kBBytes)
                                          : (uint32_t)(Cfg::kABytes + Cfg::kBBytes + Cfg::kSfaBytes);
    constexpr uint32_t kBytes = ROLE == 0   ? (uint32_t)Cfg::kABytes
                                : ROLE == 1 ? (uint32_t)Cfg::kBBytes
                                : ROLE == 2 ? (uint32_t)Cfg::kSfaBytes
                                            : (uint32_t)Cfg::kSfbBytes;
    // full[s] for the operand tiles, sf_full[s] for the scales
    auto done_bar = [&](int s) { return bar0 + 8u * ((kSf ? 3 * S : 0) + s); };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };

    const bool b_side = (ROLE == 1 || ROLE == 3);
    const uint64_t pol = b_side ? (p.b_policy == 1   ? ptx::policy_evict_first()
                                   : p.b_policy == 2 ? ptx::policy_evict_last()
                                                     : ptx::policy_evict_normal())
                                : ptx::policy_evict_last();
    uint32_t q = 0;   // position in this CTA's sequence of stages
    uint32_t issued = 0, issued_parity = 0;
    bool ok = true;
    PieceCursor<Cfg::BK, SK> cur;
    cur.start(p);
    Piece tc;
    while (ok && cur.next(p, tc)) {
        for (int it = tc.it0; it < tc.it1; ++it, ++q) {
            const int stage = (int)(q % S);
            const uint32_t phase = (q / S) & 1u;
            if (!wait_bounded(empty_bar(stage), phase ^ 1u, wctx, kRoleProducer)) {
                ok = false;
                break;
            }
            const bool drop = ROLE == 1 && p.debug_drop_stage && blockIdx.x == 0 && q == 0;
            if (!drop) {
                const uint32_t dst = base + stage * Cfg::kStageBytes + kOff;
                const uint32_t bar = done_bar(stage);
                ptx::mbar_arrive_expect_tx(bar, kBytes);
                if (ROLE == 0)
                    ptx::tma_load_3d(dst, &p.tmA[tc.g], 0, tc.bm * kBM, it * Cfg::kChunks, bar, pol);
                else if (ROLE == 1)
                    ptx::tma_load_3d(dst, &p.tmB[tc.g], 0, tc.bn * Cfg::BN, it * Cfg::kChunks, bar, pol);
                else if (ROLE == 2)
                    ptx::tma_load_3d(dst, &kp.tmSFA[tc.g], 0, it * Cfg::kMmas, tc.bm, bar, pol);
                else
                    ptx::tma_load_3d(dst, &kp.tmSFB[tc.g], 0, it * Cfg::kMmas, tc.bn * (Cfg::BN / 128),
                                     bar, pol);
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            }
        }
    }
    // copies issued but never consumed (after an abort anywhere in the CTA)
    // still land in this CTA's shared memory: wait for the last issue of
    // every slot before the CTA can exit.  On the normal path these phases
    // completed already.
    (void)ok;
    for (int s = 0; s < S; ++s)
        if (issued & (1u << s))
            wait_drain(done_bar(s), (issued_parity >> s) & 1u, wctx);
}

// L2 prefetch role (one thread): walks this CTA's stage sequence and
// prefetches each stage's B tile and B scales into L2 once the MMA thread is
// within `pf_stages` stages of it, so that more HBM reads are in flight than
// the shared-memory ring holds.  It only ever delays itself: it gives up
// (without an error) when a wait for progress exceeds the wait timeout or
// another role aborted.
template <class Cfg, bool SK>
__device__ __forceinline__ void prefetch_role(const KernelParams &kp, volatile uint32_t *progress,
                                              const WaitCtx &wctx)
{
    const GemmParams &p = kp.g;
    const uint64_t pol = p.b_policy == 1   ? ptx::policy_evict_first()
                         : p.b_policy == 2 ? ptx::policy_evict_last()
                                           : ptx::policy_evict_normal();
    PieceCursor<Cfg::BK, SK> cur;
    cur.start(p);
    Piece pc;
    uint32_t q = 0;
    while (cur.next(p, pc)) {
        for (int it = pc.it0; it < pc.it1; ++it, ++q) {
            if (q >= *progress + (uint32_t)p.pf_stages) {
                const uint64_t t0 = ptx::globaltimer_ns();
                while (q >= *progress + (uint32_t)p.pf_stages) {
                    if (*wctx.abort || ptx::globaltimer_ns() - t0 > wctx.timeout_ns)
                        return;
                    __nanosleep(128);
                }
            }
            ptx::tma_prefetch_3d(&p.tmB[pc.g], 0, pc.bn * Cfg::BN, it * Cfg::kChunks, pol);
            ptx::tma_prefetch_3d(&kp.tmSFB[pc.g], 0, it * Cfg::kMmas, pc.bn * (Cfg::BN / 128), pol);
        }
    }
}

// EPI_EX: the fused epilogue options (alpha, BF16, SwiGLU) are compiled in;
// the plain FP16 form keeps the default path's register budget.
template <class Cfg, bool EPI_EX, bool SK>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    nvfp4_group_gemm_kernel(const __grid_constant__ KernelParams kp)
{
    const GemmParams &p = kp.g;
    constexpr int BN = Cfg::BN;
    constexpr int S = Cfg::kStages;
    constexpr int EC = Cfg::kEpiCols;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);

    const uint32_t bar0 = base + Cfg::kBarOff;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto sfr_bar = [&](int s) { return bar0 + 8u * (2 * S + s); };
    auto sffull_bar = [&](int s) { return bar0 + 8u * (3 * S + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (4 * S + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (4 * S + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (4 * S + 4);
    const uint32_t sf_drain_bar = bar0 + 8u * (4 * S + 5);
    const uint32_t tmem_slot = base + Cfg::kSlotOff;
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + Cfg::kSlotOff + 4);
    volatile uint32_t *mma_progress = reinterpret_cast<volatile uint32_t *>(gbase + Cfg::kSlotOff + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full_bar(s), 2);     // the A and B loaders
            ptx::mbar_init(empty_bar(s), 1);
            ptx::mbar_init(sfr_bar(s), 1);
            ptx::mbar_init(sffull_bar(s), 2);   // the A-scale and B-scale loaders
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(accf_bar(b), 1);
            ptx::mbar_init(acce_bar(b), 4);  // lane 0 of each epilogue warp
        }
        ptx::mbar_init(drain_bar, 1);
        ptx::mbar_init(sf_drain_bar, 1);
        *abort_flag = 0u;
        *mma_progress = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(tmem_slot, Cfg::kTmemCols);
        ptx::tmem_relinquish();
        ptx::tc_fence_before();
    }
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = ptx::ld_shared_u32(tmem_slot);
    // With a programmatic launch the set-up above overlaps the previous
    // kernel; nothing below touches global memory before that kernel is done,
    // except the A and B loads of an early_ab launch (the previous kernel is
    // then the library's scale relayout, which reads neither).
    if (!(p.early_ab && (warp == kFirstLoaderWarp || warp == kFirstLoaderWarp + 1)))
        ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();

    const WaitCtx wctx{abort_flag, p.err, p.timeout_ns};
    if (warp == Cfg::kPrefetchWarp) {
        if (lane == 0 && p.pf_stages > 0)
            prefetch_role<Cfg, SK>(kp, mma_progress, wctx);
    } else if (warp >= kFirstLoaderWarp) {
        if (lane == 0) {
            switch (warp - kFirstLoaderWarp) {
            case 0: loader_role<Cfg, SK, 0>(kp, base, bar0, wctx); break;
            case 1: loader_role<Cfg, SK, 1>(kp, base, bar0, wctx); break;
            case 2: loader_role<Cfg, SK, 2>(kp, base, bar0, wctx); break;
            default: loader_role<Cfg, SK, 3>(kp, base, bar0, wctx); break;
            }
        }
    } else if (warp == kSfWarp) {
        if (lane == 0) {
            // ------------------------------------------- scale copies
            // once a stage's scales have landed, copy the atoms into the
            // slot's own tensor-memory columns and signal sf_ready[slot]
            uint32_t q = 0;
            bool ok = true, issued_any = false;
            PieceCursor<Cfg::BK, SK> cur;
            cur.start(p);
            Piece tc;
            while (ok && cur.next(p, tc)) {
                const int kchunks = p.kchunks[tc.g];
                for (int it = tc.it0; it < tc.it1; ++it, ++q) {
                    const int stage = (int)(q % S);
                    if (!wait_bounded(sffull_bar(stage), (q / S) & 1u, wctx, kRoleSf)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const int nk = kblocks_in_stage<Cfg::BK>(kchunks, it);
                    const uint32_t ssfa = base + stage * Cfg::kStageBytes + Cfg::kABytes + Cfg::kBBytes;
                    const uint32_t ssfb = ssfa + Cfg::kSfaBytes;
#pragma unroll
                    for (int j = 0; j < Cfg::kMmas; ++j) {
                        if (j < nk) {
                            ptx::tc_cp_32x128b_warpx4(tmem_base + Cfg::sfa_col(stage, j),
                                                      desc_scale_atom(ssfa + 512 * j));
#pragma unroll
                            for (int h = 0; h < BN / 128; ++h)
                                ptx::tc_cp_32x128b_warpx4(
                                    tmem_base + Cfg::sfb_col(stage, j, h),
                                    desc_scale_atom(ssfb + Cfg::kMmas * 512 * h + 512 * j));
                        }
                    }
                    ptx::tc_commit(sfr_bar(stage));
                    issued_any = true;
                }
            }
            if (issued_any) {   // copies in flight write tensor memory: wait for them
                ptx::tc_commit(sf_drain_bar);
                wait_drain(sf_drain_bar, 0u, wctx);
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            uint32_t q = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true, issued_any = false;
            PieceCursor<Cfg::BK, SK> cur;
            cur.start(p);
            Piece tc;
            while (ok && cur.next(p, tc)) {
                const int kchunks = p.kchunks[tc.g];
                if (!wait_bounded(acce_bar(acc), acc_phase ^ 1u, wctx, kRoleMma)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int it = tc.it0; it < tc.it1; ++it, ++q) {
                    const int stage = (int)(q % S);
                    if (!wait_bounded(full_bar(stage), (q / S) & 1u, wctx, kRoleMma) ||
                        !wait_bounded(sfr_bar(stage), (q / S) & 1u, wctx, kRoleMma)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const int nk = kblocks_in_stage<Cfg::BK>(kchunks, it);
                    const uint32_t sa = base + stage * Cfg::kStageBytes;
                    const uint32_t sb = sa + Cfg::kABytes;
#pragma unroll
                    for (int j = 0; j < Cfg::kMmas; ++j) {
                        if (j < nk) {
                            // MMA j reads bytes [32 (j % 4), +32) of every row of chunk j / 4
                            const uint32_t koff_a = (j / 4) * kBM * 128 + (j % 4) * 32;
                            const uint32_t koff_b = (j / 4) * BN * 128 + (j % 4) * 32;
                            ptx::tc_mma_nvfp4(d_tmem, desc_operand_sw128(sa + koff_a),
                                              desc_operand_sw128(sb + koff_b), Cfg::kIdesc,
                                              tmem_base + Cfg::sfa_col(stage, j),
                                              tmem_base + Cfg::sfb_col(stage, j, 0),
                                              (it > tc.it0 || j > 0) ? 1u : 0u);
                        }
                    }
                    // frees the slot once these MMAs (and, through sf_ready,
                    // the scale copies before them) are complete
                    ptx::tc_commit(empty_bar(stage));
                    issued_any = true;
                    *mma_progress = q + 1;   // paces the L2 prefetcher
                }
                if (!ok)
                    break;
                ptx::tc_commit(accf_bar(acc));
                if (++acc == Cfg::kAccBufs) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (issued_any) {
                // tensor-core work in flight still reads shared memory and
                // writes tensor memory: wait for all of it before teardown
                ptx::tc_commit(drain_bar);
                wait_drain(drain_bar, 0u, wctx);
            }
        }
    } else if (warp < 4) {
        // ---------------------------------------------------- epilogue
        int acc = 0;
        uint32_t acc_phase = 0;
        int sbuf = 0;
        const uint32_t stage_buf = base + Cfg::kEpiOff + warp * Cfg::kEpiBufs * Cfg::kEpiBufBytes;
        const uint32_t lane_tmem = (uint32_t)(warp * 32) << 16;
        const int row = warp * 32 + lane;   // accumulator row (tensor-memory lane) of this thread
        uint32_t epoch = 0;                 // stream-K: the launch's flag value
        if constexpr (SK)
            epoch = *reinterpret_cast<volatile const uint32_t *>(p.sk_epoch);
        PieceCursor<Cfg::BK, SK> cur;
        cur.start(p);
        Piece tc;
        while (cur.next(p, tc)) {
            // lane 0 waits; the outcome is broadcast so the warp stays
            // converged for the .sync.aligned tensor-memory loads
            uint32_t ready = 1u;
            if (lane == 0)
                ready = wait_bounded(accf_bar(acc), acc_phase, wctx, kRoleEpilogue) ? 1u : 0u;
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (!ready)
                break;
            ptx::tc_fence_after();
            const int M = p.M[tc.g];
            const int N = p.N[tc.g];
            const int m0 = tc.bm * kBM + warp * 32;
            const int n0 = tc.bn * BN;
            const uint32_t acc_taddr = tmem_base + lane_tmem + acc * BN;
            if constexpr (SK) {
                if (tc.it0 > 0) {
                    // a later part of a tile that another CTA owns: the
                    // partial sum goes to this CTA's slot, the accumulator
                    // back to the MMA thread, then the flag is published
                    if (m0 < M)
                        store_partial<BN>(p.sk_ws, acc_taddr, n0, N, row);
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        ptx::mbar_arrive(acce_bar(acc));
                    if (m0 < M) {
                        __threadfence();
                        __syncwarp();
                        if (lane == 0)
                            ptx::st_release_gpu(p.sk_flags + blockIdx.x * 4 + warp, epoch);
                    }
                    if (++acc == Cfg::kAccBufs) {
                        acc = 0;
                        acc_phase ^= 1u;
                    }
                    continue;
                }
            }
            // stream-K owner of a cut tile (it holds the tile's first stages):
            // the CTAs after this one whose ranges start inside the tile hold
            // the rest of its sum; their ranges began with it, so their flags
            // are normally set long before
            int h0 = 0, h1 = 0;
            if constexpr (SK) {
                if (tc.it1 < tc.nst && m0 < M) {
                    h0 = (int)blockIdx.x + 1;
                    h1 = h0;
                    while (h1 < (int)gridDim.x && sk_begin(p, h1) < tc.u1)
                        ++h1;
                    uint32_t ok = 1u;
                    if (lane == 0)
                        for (int hc = h0; hc < h1 && ok; ++hc)
                            ok = wait_flag_bounded(p.sk_flags + hc * 4 + warp, epoch, wctx) ? 1u : 0u;
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok)
                        break;
                    __syncwarp();
                    __threadfence();
                }
            }
            // 1. this thread's whole accumulator row -> 16-bit output pairs in
            // registers
            uint32_t h[BN / 2];
            if (m0 < M)
                epilogue_load<BN, EPI_EX, SK>(p, tc.g, acc_taddr, n0, N, h, h0, h1, row);
            // 2. every lane's loads have completed (wait::ld): the accumulator
            // goes back to the MMA thread before the stores start, so the next
            // tile's MMAs overlap them
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(acce_bar(acc));
            // 3. swizzled shared staging + TMA tensor stores, EC columns each
            const bool sw = EPI_EX && p.swiglu;
            const int on0 = sw ? n0 / 2 : n0;     // output columns
            const int oN = sw ? N / 2 : N;
            const int ocols = sw ? BN / 2 : BN;
            // the CTA's last tile: every MMA has completed and no load is
            // left, so the operand ring is free -- each chunk gets its own
            // staging buffer there and the stores go out back to back
            const bool last_tile = cur.done(p);
            const uint32_t ring_buf = base + (uint32_t)(warp * (BN / EC)) * Cfg::kEpiBufBytes;
            if (m0 < M && last_tile && p.c_wide[tc.g]) {
                store_slab_wide<BN>(&p.tmCw[tc.g], base + (uint32_t)(warp * (BN / 64)) * 4096u, lane, on0, oN,
                                    ocols, m0, h);
            } else if (m0 < M) {
#pragma unroll
                for (int c = 0; c < BN / EC; ++c) {
                    if (c * EC < ocols && on0 + c * EC < oN) {   // warp-uniform
                        // the store that last used this buffer must have
                        // finished reading it
                        if (lane == 0 && !last_tile) {
                            if constexpr (Cfg::kEpiBufs == 2)
                                ptx::bulk_wait_group_read<1>();
                            else
                                ptx::bulk_wait_group_read<0>();
                        }
                        __syncwarp();
                        const uint32_t buf =
                            last_tile ? ring_buf + c * Cfg::kEpiBufBytes : stage_buf + sbuf * Cfg::kEpiBufBytes;
                        // one row of EC halves per lane; 16-byte chunk q of row
                        // r sits at chunk q ^ (swizzle phase of r), the pattern
                        // of the C tensor map's EC*2-byte swizzle
                        // (conflict-free)
                        constexpr int kQ = EC / 8;
                        const uint32_t row = buf + lane * (EC * 2);
                        const int phase_r = (EC == 64) ? (lane & 7) : ((lane >> 1) & 3);
#pragma unroll
                        for (int q = 0; q < kQ; ++q)
                            ptx::st_shared_v4(row + ((q ^ phase_r) << 4), h[c * (EC / 2) + 4 * q],
                                              h[c * (EC / 2) + 4 * q + 1], h[c * (EC / 2) + 4 * q + 2],
                                              h[c * (EC / 2) + 4 * q + 3]);
                        ptx::fence_proxy_async_shared();
                        __syncwarp();
                        if (lane == 0) {
                            ptx::tma_store_2d(&p.tmC[tc.g], buf, on0 + c * EC, m0);
                            ptx::bulk_commit_group();
                        }
                        __syncwarp();
                        if constexpr (Cfg::kEpiBufs == 2)
                            sbuf ^= 1;
                    }
                }
            }
            if (++acc == Cfg::kAccBufs) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0)
            ptx::bulk_wait_group<0>();
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
    if constexpr (SK) {
        // the last CTA to finish moves the epoch on (and re-arms the count),
        // so the next launch -- which reads both only after this grid has
        // completed -- never mistakes this launch's flags for its own
        if (threadIdx.x == 0) {
            __threadfence();
            if (atomicAdd(p.sk_epoch + 1, 1u) == gridDim.x - 1) {
                volatile uint32_t *ep = p.sk_epoch;
                ep[1] = 0u;
                ep[0] = ep[0] + 1u;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Kernel configurations, chosen per call by the host (group_gemm.cu).
//   CfgStream:  BN = 128, 512-K stages (256 contiguous bytes per row per
//               load), 3 stages, two accumulators, one 2 KiB staging buffer
//               per epilogue warp
//   CfgWide:    BN = 256 -- half the A re-reads -- 256-K stages, 4 stages,
//               one accumulator
//   CfgWide512: BN = 256 with 512-K stages, 2 stages
//   CfgCompute: BN = 128, 256-K stages, 4 stages, two 4 KiB staging buffers
//               per warp (64-column stores)
// ---------------------------------------------------------------------------
using CfgStream = GemmConfig<128, 512, 3, 32, 1>;
using CfgWide = GemmConfig<256, 256, 4, 32, 1>;
using CfgWide512 = GemmConfig<256, 512, 2, 32, 1>;
using CfgCompute = GemmConfig<128, 256, 4, 64, 2>;

}  // namespace nvfp4
