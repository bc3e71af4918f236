// Input projection of one LSTM layer, both directions in one launch:
//     G[m][n] = sum_k X[m][k] * Wp[n][k],   m < rows, n < 1024,
// the dense `x . W^T` over every step of every window that the speakrs 0.6.0
// pages run per layer before the recurrence (lstmproj.rs module docs;
// `InputProjection::enqueue`), with the gate columns already in the packed,
// unit-interleaved order (the packer reorders W's rows).
//
// Design (sm_103a), a persistent kernel, one CTA per SM:
//  * CTA b walks tiles b, b + grid, ... of 128 rows x 256 gate columns of G
//    (tile t: rows 128*(t/4), columns 256*(t%4)), so the CTAs running
//    together read the same rows of X from L2; each CTA loads its whole W
//    tile itself (W is 1-2 MiB per layer and stays in L2), so no CTA writes
//    into another CTA's shared memory and the kernel needs no cluster;
//  * K advances in blocks of 16 fp32 (64 bytes, 64-byte swizzle) through a
//    192 KiB shared-memory ring: 4 stages of 48 KiB (X, X lo, W hi, W lo) in
//    3xTF32, 8 stages of 24 KiB in the single-product mode; with few rows
//    (the 256-column grid would fill at most half the SMs) the tiles are 128
//    columns wide, twice as many CTAs;
//  * warp 8 (TMA producer) loads the X block and the TF32 hi and lo planes of
//    the W tile (split on the host) into the ring; a stage is reused only
//    once the MMAs that read it have completed;
//  * warps 0-3 split the X block in place into its TF32 hi part and a second
//    buffer with the TF32 lo remainder;
//  * one thread of warp 9 issues tcgen05.mma kind::tf32 (M=128, N=256, K=8)
//    into one of two tensor-memory accumulators (2 x 256 columns):
//    x_hi*w_hi + x_hi*w_lo + x_lo*w_hi, the 3xTF32 split that keeps fp32-level
//    accuracy (TF32 alone was not accurate enough on some parts, per the
//    pages' `tf32_projection_accurate`).  The single-product TF32 mode (the
//    pages' `CudaMath::Tf32`) issues x_hi*w_hi alone: the lo plane of W is
//    neither loaded nor used and the converters only round X to TF32;
//  * warps 4-7 (epilogue) read a finished accumulator with tcgen05.ld, write
//    32-column slices of their 32 rows into a double-buffered shared-memory
//    staging area (128-byte swizzle, conflict-free) and hand each 4 KiB
//    slice to the TMA engine as one bulk tensor store, while the MMA fills
//    the other accumulator; the slices go out paced by the MMA's progress
//    through the next tile.
// Every mbarrier wait is bounded in time; a wait that runs out sets a bit in
// the fault word, every role stops, and the CTA drains its TMA loads and MMAs
// before it frees tensor memory and returns.
#include <cudaTypedefs.h>
#include <mutex>

#include "common.cuh"

namespace lstm {
namespace {

constexpr int BM = 128;  // rows per tile (MMA M)
constexpr int BK = 16;   // fp32 per K block = 64 bytes
constexpr int A_BYTES = BM * BK * 4;                     // 8 KiB
// Shared memory: [resident W tile] [K-block stage ring] [the epilogue's
// store staging: 4 warps x 2 slices of 4 KiB] [barriers]; 224 KiB of data.
constexpr int DATA_BYTES = 224 * 1024;
constexpr int OUT_COLS = 32;                             // columns per store slice
constexpr int OUT_BYTES = 32 * OUT_COLS * 4;             // one warp's 32 rows: 4 KiB
constexpr int OUT_OFFSET = DATA_BYTES - 4 * 2 * OUT_BYTES;
constexpr int MAX_STAGES = 8;
constexpr int CONVERTERS = 128;                          // warps 0-3
constexpr int EPILOGUE = 128;                            // warps 4-7
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int THREADS = 320;
constexpr size_t SMEM_BYTES = DATA_BYTES + 1024 + 256;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s
// K blocks a resident W tile holds: K <= 64 (the first layer's 60 inputs)
constexpr int RESIDENT_KBLOCKS = 4;

// One instantiation: tiles of BN gate columns, 3xTF32 or single products.
// RESIDENT_W (K <= 64): a CTA's W tile stays in shared memory for all its
// tiles and the ring carries only X.  With 4 K blocks per tile, reloading
// the 128 KiB W tile (hi and lo) for every 128-row tile made the loads, not
// the tensor pipe, the limit.  The grid is then a multiple of the column
// tiles, so a CTA's tiles t, t + grid, ... share one column tile.
template <int BN_, bool SINGLE_, bool RESIDENT_W_ = false>
struct Shape {
    static constexpr int BN = BN_;  // MMA N: output columns per tile
    static constexpr bool SINGLE = SINGLE_;
    static constexpr bool RESIDENT_W = RESIDENT_W_;
    static constexpr int B_BYTES = BN * BK * 4;
    static constexpr int PLANES = SINGLE ? 1 : 2;                // W hi (and lo)
    static constexpr int W_RES_BYTES = RESIDENT_W ? RESIDENT_KBLOCKS * PLANES * B_BYTES : 0;
    static constexpr int RING_BYTES = OUT_OFFSET - W_RES_BYTES;
    // 3xTF32 keeps A hi, A lo, B hi, B lo per stage; the single-product
    // mode only A hi and B hi, so the same ring holds twice the K blocks;
    // with a resident W the stages hold only A
    static constexpr int A_STAGE_BYTES = SINGLE ? A_BYTES : 2 * A_BYTES;
    static constexpr int STAGE_BYTES = A_STAGE_BYTES + (RESIDENT_W ? 0 : PLANES * B_BYTES);
    static constexpr int STAGES =
        RING_BYTES / STAGE_BYTES < MAX_STAGES ? RING_BYTES / STAGE_BYTES : MAX_STAGES;
    static constexpr int A_LO = A_BYTES;                         // 3xTF32 only
    static constexpr int B_HI = A_STAGE_BYTES;                   // in the stage (not RESIDENT_W)
    static constexpr int B_LO = B_HI + B_BYTES;                  // 3xTF32 only
    static constexpr uint32_t TX_BYTES = A_BYTES + (RESIDENT_W ? 0 : PLANES * B_BYTES);
    static constexpr uint32_t ACC_COLS = BN;                     // per accumulator
    static constexpr uint32_t TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;  // two accumulators
    static constexpr int TILES_N = kGateColumns / BN;
    static constexpr uint32_t IDESC = ptx::tf32_idesc(BM, BN);
    static_assert(STAGE_BYTES % 1024 == 0 && BN % 16 == 0 && BN <= 256 && STAGES >= 4 &&
                      W_RES_BYTES % 1024 == 0,
                  "tile shape");
};
using GatesShape = Shape<256, false>;
using GatesTf32Shape = Shape<256, true>;
using GatesNarrowShape = Shape<128, false>;  // few rows: twice the tiles
using GatesResidentShape = Shape<256, false, true>;        // K <= 64
using GatesTf32ResidentShape = Shape<256, true, true>;     // K <= 64
using GatesNarrowResidentShape = Shape<128, false, true>;  // K <= 64
static_assert(GatesShape::BN == kProjectionWBoxRows && BM == kProjectionBoxRows &&
                  GatesNarrowShape::BN == kProjectionNarrowWBoxRows,
              "TMA boxes");

using ptx::sw64_desc;
using ptx::split4;

// Waits without regard to the abort flag (used to drain in-flight work).
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity, unsigned *fault)
{
    ptx::mbar_wait_drain(bar, parity, fault, WAIT_LIMIT_NS);
}

template <class S>
__global__ void __launch_bounds__(THREADS, 1)
projection_kernel(const __grid_constant__ CUtensorMap x_map,
                  const __grid_constant__ CUtensorMap whi_map,
                  const __grid_constant__ CUtensorMap wlo_map,
                  const __grid_constant__ CUtensorMap out_map, int rows, int kblocks, int tiles,
                  unsigned *fault, unsigned long long wait_limit_ns, int withhold)
{
    using RG = S;
    constexpr bool SINGLE = S::SINGLE;
    constexpr int STAGES = S::STAGES;
    constexpr int STAGE_BYTES = S::STAGE_BYTES;
    constexpr int BN = S::BN;
    constexpr int TILES_N = S::TILES_N;
    constexpr uint32_t ACC_COLS = S::ACC_COLS;
    constexpr uint32_t IDESC = S::IDESC;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + DATA_BYTES);
    uint64_t *conv = full + MAX_STAGES;
    uint64_t *empty = conv + MAX_STAGES;
    uint64_t *acc_full = empty + MAX_STAGES;  // [2]
    uint64_t *acc_empty = acc_full + 2;       // [2]
    uint64_t *w_full = acc_empty + 2;         // the resident W tile landed (RESIDENT_W)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(w_full + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *progress = abort_flag + 1;  // K blocks whose MMAs were issued

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&conv[s], CONVERTERS);
            ptx::mbar_init(&empty[s], 1);  // the MMAs that read the stage completed
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&acc_full[a], 1);
            ptx::mbar_init(&acc_empty[a], EPILOGUE);
        }
        ptx::mbar_init(w_full, 1);
        *abort_flag = 0;
        *progress = 0;
        ptx::fence_mbar_init();
    }
    if (warp == PRODUCER_WARP && lane == 0) {
        ptx::prefetch_tensormap(&x_map);
        ptx::prefetch_tensormap(&whi_map);
        ptx::prefetch_tensormap(&wlo_map);
        ptx::prefetch_tensormap(&out_map);
    }
    if (warp == MMA_WARP) {
        ptx::tmem_alloc(tmem_slot, S::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    // Programmatic dependent launch: the set-up above overlaps the tail of
    // the kernel before this one; X (that kernel's output) and G (which it
    // may still read) are touched only after it has completed.
    ptx::griddep_wait();
    // ... and the recurrence after this one may be scheduled now (on the SMs
    // this grid leaves free); it waits for this grid's end before it reads G
    ptx::griddep_launch_dependents();
    const uint32_t tmem = *tmem_slot;
    const int first = static_cast<int>(blockIdx.x);
    const int stride = static_cast<int>(gridDim.x);
    long issued = 0;            // producer: K blocks whose loads were issued
    bool w_issued = false;      // producer: the resident W tile's loads were issued
    uint8_t *const ring = smem + S::W_RES_BYTES;
    int committed_tiles = 0;    // MMA: accumulators committed

    if (warp == PRODUCER_WARP) {
        // failure test (`withhold`): nothing is loaded, so the converters'
        // waits run out
        if (lane == 0 && !withhold) {
            if constexpr (S::RESIDENT_W) {
                // this CTA's column tile, all its K blocks, once
                const int n0 = (first % TILES_N) * BN;
                ptx::mbar_arrive_expect_tx(w_full, kblocks * S::PLANES * S::B_BYTES);
                for (int kb = 0; kb < kblocks; ++kb) {
                    ptx::tma_load_2d(smem + kb * S::B_BYTES, &whi_map, w_full, kb * BK, n0);
                    if constexpr (!SINGLE)
                        ptx::tma_load_2d(smem + (RESIDENT_KBLOCKS + kb) * S::B_BYTES, &wlo_map,
                                         w_full, kb * BK, n0);
                }
                w_issued = true;
            }
            long kbi = 0;
            for (int t = first; t < tiles && !*abort_flag; t += stride) {
                const int m0 = (t / TILES_N) * BM;
                const int n0 = (t % TILES_N) * BN;
                for (int kb = 0; kb < kblocks; ++kb, ++kbi) {
                    const int s = static_cast<int>(kbi % STAGES);
                    const uint32_t n = static_cast<uint32_t>(kbi / STAGES);
                    if (n > 0 && !ptx::mbar_wait_bounded(&empty[s], (n - 1) & 1, abort_flag, fault,
                                                         kFaultProducer, wait_limit_ns))
                        break;
                    uint8_t *st = ring + s * STAGE_BYTES;
                    ptx::mbar_arrive_expect_tx(&full[s], RG::TX_BYTES);
                    ptx::tma_load_2d(st, &x_map, &full[s], kb * BK, m0);
                    if constexpr (!S::RESIDENT_W) {
                        ptx::tma_load_2d(st + RG::B_HI, &whi_map, &full[s], kb * BK, n0);
                        if constexpr (!SINGLE)
                            ptx::tma_load_2d(st + RG::B_LO, &wlo_map, &full[s], kb * BK, n0);
                    }
                    issued = kbi + 1;
                }
            }
        }
    } else if (warp == MMA_WARP) {
        if (lane == 0) {
            long kbi = 0;
            int ti = 0;
            // the resident W tile has landed (its wait, like every other, is
            // bounded: a failure here skips the tile loop)
            const bool w_ok = !S::RESIDENT_W ||
                              ptx::mbar_wait_bounded(w_full, 0, abort_flag, fault, kFaultMma,
                                                     wait_limit_ns);
            for (int t = first; w_ok && t < tiles && !*abort_flag; t += stride, ++ti) {
                const int a = ti & 1;
                const uint32_t use = static_cast<uint32_t>(ti >> 1);
                if (use > 0 && !ptx::mbar_wait_bounded(&acc_empty[a], (use - 1) & 1, abort_flag,
                                                       fault, kFaultMma, wait_limit_ns))
                    break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(a) * ACC_COLS;
                bool ok = true;
                for (int kb = 0; kb < kblocks; ++kb, ++kbi) {
                    const int s = static_cast<int>(kbi % STAGES);
                    const uint32_t n = static_cast<uint32_t>(kbi / STAGES);
                    if (!ptx::mbar_wait_bounded(&conv[s], n & 1, abort_flag, fault, kFaultMma,
                                                wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a_hi = ptx::smem_u32(ring + s * STAGE_BYTES);
                    const uint32_t a_lo = a_hi + RG::A_LO;
                    const uint32_t w_res = ptx::smem_u32(smem);
                    const uint32_t b_hi = S::RESIDENT_W
                                              ? w_res + static_cast<uint32_t>(kb * S::B_BYTES)
                                              : a_hi + RG::B_HI;
                    const uint32_t b_lo =
                        S::RESIDENT_W
                            ? w_res + static_cast<uint32_t>((RESIDENT_KBLOCKS + kb) * S::B_BYTES)
                            : a_hi + RG::B_LO;
#pragma unroll
                    for (int j = 0; j < BK / 8; ++j) {
                        const uint32_t off = j * 32;  // 8 TF32 = 32 bytes along K
                        ptx::mma_tf32(d_tmem, sw64_desc(a_hi + off), sw64_desc(b_hi + off), IDESC,
                                      (kb | j) != 0);
                        if constexpr (!SINGLE) {
                            ptx::mma_tf32(d_tmem, sw64_desc(a_hi + off), sw64_desc(b_lo + off),
                                          IDESC, 1);
                            ptx::mma_tf32(d_tmem, sw64_desc(a_lo + off), sw64_desc(b_hi + off),
                                          IDESC, 1);
                        }
                    }
                    ptx::mma_commit(&empty[s]);
                    *progress = static_cast<int>(kbi + 1);
                }
                ptx::mma_commit(&acc_full[a]);  // also when stopping early: frees the epilogue
                committed_tiles = ti + 1;
                if (!ok)
                    break;
            }
        }
    } else if (warp < 4) {
        // converters: split X into TF32 hi (in place) and lo; the
        // single-product mode only rounds X to TF32 in place
        const int tid = threadIdx.x;
        long kbi = 0;
        for (int t = first; t < tiles && !*abort_flag; t += stride) {
            bool ok = true;
            for (int kb = 0; kb < kblocks; ++kb, ++kbi) {
                const int s = static_cast<int>(kbi % STAGES);
                const uint32_t n = static_cast<uint32_t>(kbi / STAGES);
                if (!ptx::mbar_wait_bounded(&full[s], n & 1, abort_flag, fault, kFaultConverter,
                                            wait_limit_ns)) {
                    ok = false;
                    break;
                }
                float4 *a = reinterpret_cast<float4 *>(ring + s * STAGE_BYTES);
                float4 *alo = reinterpret_cast<float4 *>(ring + s * STAGE_BYTES + RG::A_LO);
                if constexpr (SINGLE) {
#pragma unroll
                    for (int i = 0; i < A_BYTES / 16 / CONVERTERS; ++i) {
                        const int idx = tid + i * CONVERTERS;
                        const float4 v = a[idx];
                        a[idx] = make_float4(ptx::tf32_rna(v.x), ptx::tf32_rna(v.y),
                                             ptx::tf32_rna(v.z), ptx::tf32_rna(v.w));
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < A_BYTES / 16 / CONVERTERS; ++i) {
                        const int idx = tid + i * CONVERTERS;
                        float4 hi, lo;
                        split4(a[idx], hi, lo);
                        a[idx] = hi;
                        alo[idx] = lo;
                    }
                }
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive(&conv[s]);
            }
            if (!ok)
                break;
        }
    } else if (warp >= 4) {
        // epilogue: warp 4+q reads TMEM lanes 32q .. 32q+31 (warp id mod 4 = q)
        const int q = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        uint8_t *stage_out = smem + OUT_OFFSET + q * 2 * OUT_BYTES;
        int slices = 0;  // store slices this warp issued
        int ti = 0;
        for (int t = first; t < tiles; t += stride, ++ti) {
            const int a = ti & 1;
            const uint32_t use = static_cast<uint32_t>(ti >> 1);
            bool got = ptx::mbar_wait_bounded(&acc_full[a], use & 1, abort_flag, fault,
                                              kFaultEpilogue, wait_limit_ns);
            // tcgen05.ld is warp-collective: continue only if every lane may
            if (!__all_sync(0xffffffffu, got) || *abort_flag)
                break;
            ptx::tc_fence_after();
            const int m0 = (t / TILES_N) * BM + q * 32;  // this warp's rows
            const int n0 = (t % TILES_N) * BN;
            const uint32_t acc = tmem + lane_base + static_cast<uint32_t>(a) * ACC_COLS;
            // Pace the stores: slice c of this tile goes out once the next
            // tile's mainloop has issued c/NSLICE of its K blocks, so G
            // streams to memory under the next tile's compute instead of
            // every CTA writing its whole tile at once and stalling the loads.
            // With a resident W tile the ring carries only X and a tile has
            // 4 K blocks, so the stores go out unpaced (measured: 3.5 % faster
            // at 150 784 rows, no change at fewer).
            constexpr int NSLICE = BN / OUT_COLS;
            const bool paced = !S::RESIDENT_W && t + stride < tiles;
            const long next_kb = static_cast<long>(ti + 1) * kblocks;
#pragma unroll 1
            for (int c = 0; c < NSLICE; ++c, ++slices) {
                if (paced) {
                    const long want = next_kb + (static_cast<long>(c) * kblocks) / NSLICE;
                    if (*progress < want && !*abort_flag) {
                        const uint64_t start = ptx::globaltimer();
                        while (*progress < want && !*abort_flag &&
                               ptx::globaltimer() - start < wait_limit_ns)
                            __nanosleep(64);
                    }
                }
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(acc + c * OUT_COLS, r);
                ptx::tmem_ld_wait();
                // the store that last used this buffer (two slices ago) has read it
                uint8_t *buf = stage_out + (slices & 1) * OUT_BYTES;
                if (lane == 0)
                    ptx::bulk_wait_group_read<1>();
                __syncwarp();
                // lane = row; 16-byte chunk j of the row goes to chunk j ^ (row % 8)
                float4 *row = reinterpret_cast<float4 *>(buf + lane * (OUT_COLS * 4));
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    row[j ^ (lane & 7)] =
                        make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                    __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (m0 < rows)
                        ptx::tma_store_2d(&out_map, buf, n0 + c * OUT_COLS, m0);
                    ptx::bulk_commit_group();
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&acc_empty[a]);
        }
        // the staging buffers stay valid until the stores have completed
        if (lane == 0)
            ptx::bulk_wait_group<0>();
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == PRODUCER_WARP && lane == 0) {
        // every issued TMA load has landed before the CTA's shared memory goes away
        for (long kb = issued - STAGES < 0 ? 0 : issued - STAGES; kb < issued; ++kb)
            drain_wait(&full[kb % STAGES], static_cast<uint32_t>(kb / STAGES) & 1, fault);
        if (w_issued)
            drain_wait(w_full, 0, fault);
    }
    if (warp == MMA_WARP) {
        if (lane == 0) {
            // every MMA has completed before tensor memory is freed
            for (int ti = committed_tiles - 2 < 0 ? 0 : committed_tiles - 2; ti < committed_tiles; ++ti)
                drain_wait(&acc_full[ti & 1], static_cast<uint32_t>(ti >> 1) & 1, fault);
        }
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, S::TMEM_COLS);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

int g_max_ctas[64] = {};  // CTAs of the projection a device runs at once

} // namespace

namespace {
int encode_map(CUtensorMap *map, const float *base, long rows, int cols, int box_cols,
               int box_rows, CUtensorMapSwizzle swizzle)
{
    auto encode = encode_fn();
    if (!encode)
        return fail(LSTM_E_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    if ((reinterpret_cast<uintptr_t>(base) & 15) != 0)
        return fail(LSTM_E_INVALID, "matrix base %p is not 16-byte aligned", (const void *)base);
    if ((cols * 4) % 16 != 0)
        return fail(LSTM_E_INVALID, "row pitch %d bytes is not a multiple of 16", cols * 4);
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(LSTM_E_CUDA, "cuTensorMapEncodeTiled failed (%d) for %ld x %d", (int)r, rows,
                    cols);
    return LSTM_OK;
}
}  // namespace

int encode_matrix_map(CUtensorMap *map, const float *base, long rows, int cols, int box_rows)
{
    return encode_map(map, base, rows, cols, BK, box_rows, CU_TENSOR_MAP_SWIZZLE_64B);
}

int encode_store_map(CUtensorMap *map, float *base, long rows, int cols)
{
    return encode_map(map, base, rows, cols, OUT_COLS, 32, CU_TENSOR_MAP_SWIZZLE_128B);
}

namespace {
// Every instantiation, for the per-device attributes.
const void *const kKernels[] = {
    reinterpret_cast<const void *>(&projection_kernel<GatesShape>),
    reinterpret_cast<const void *>(&projection_kernel<GatesTf32Shape>),
    reinterpret_cast<const void *>(&projection_kernel<GatesNarrowShape>),
    reinterpret_cast<const void *>(&projection_kernel<GatesResidentShape>),
    reinterpret_cast<const void *>(&projection_kernel<GatesTf32ResidentShape>),
    reinterpret_cast<const void *>(&projection_kernel<GatesNarrowResidentShape>),
};

// Persistent grid over the row tiles (128 rows) times S::TILES_N column
// tiles, no larger than what runs at once.
template <class S>
int launch_tiles(const CUtensorMap &x_map, const CUtensorMap &whi_map,
                 const CUtensorMap &wlo_map, const CUtensorMap &out_map, int rows, int kp,
                 unsigned *fault, cudaStream_t stream, int *grid_out)
{
    if (rows <= 0 || kp <= 0 || kp % 32 != 0)
        return fail(LSTM_E_INVALID, "tensor-core GEMM: rows %d, kp %d", rows, kp);
    const long mtiles = (static_cast<long>(rows) + BM - 1) / BM;
    const long tiles = mtiles * S::TILES_N;
    if (tiles > 0x7fffffffL)
        return fail(LSTM_E_OVERFLOW, "tensor-core GEMM: %d rows", rows);
    int dev = 0;
    int st = cuda_status(cudaGetDevice(&dev), "current device");
    if (st != LSTM_OK)
        return st;
    int fit = (dev >= 0 && dev < 64 && g_max_ctas[dev] > 0) ? g_max_ctas[dev] : 148;
    if (S::RESIDENT_W) {
        // a CTA's tiles (first, first + grid, ...) must share a column tile
        if (kp > RESIDENT_KBLOCKS * BK)
            return fail(LSTM_E_INVALID, "tensor-core GEMM: kp %d above the resident W tile", kp);
        fit -= fit % S::TILES_N;
    }
    const long grid = tiles < fit ? tiles : fit;
    if (grid_out)
        *grid_out = static_cast<int>(grid);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int kblocks = kp / BK;
    const int ntiles = static_cast<int>(tiles);
    const KernelTest test = kernel_test(kTestProjection);
    if ((st = check_launch_injection("tensor-core GEMM launch")))
        return st;
    return cuda_status(cudaLaunchKernelEx(&cfg, projection_kernel<S>, x_map, whi_map, wlo_map,
                                          out_map, rows, kblocks, ntiles, fault,
                                          test.wait_limit_ns, test.withhold),
                       "tensor-core GEMM launch");
}
}  // namespace

int projection_prepare(int device)
{
    if (device < 0 || device >= 64)
        return fail(LSTM_E_INVALID, "device %d out of range", device);
    int sms = 0;
    int st = cuda_status(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device),
                         "SM count");
    if (st != LSTM_OK)
        return st;
    for (const void *fn : kKernels) {
        st = cuda_status(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(SMEM_BYTES)),
                         "projection shared-memory attribute");
        if (st != LSTM_OK)
            return st;
    }
    // the persistent grid is no larger than what runs at once (every
    // instantiation has the same block and shared-memory size)
    int per_sm = 0;
    st = cuda_status(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                         &per_sm, projection_kernel<GatesShape>, THREADS, SMEM_BYTES),
                     "projection occupancy");
    if (st != LSTM_OK)
        return st;
    g_max_ctas[device] = per_sm > 0 ? per_sm * sms : sms;
    return LSTM_OK;
}

int encode_projection_w(ProjectionW *w, const float *wp_hi, const float *wp_lo, int kp)
{
    int st;
    if ((st = encode_matrix_map(&w->hi, wp_hi, kGateColumns, kp, kProjectionWBoxRows)) ||
        (st = encode_matrix_map(&w->lo, wp_lo, kGateColumns, kp, kProjectionWBoxRows)) ||
        (st = encode_matrix_map(&w->hi_narrow, wp_hi, kGateColumns, kp,
                                kProjectionNarrowWBoxRows)) ||
        (st = encode_matrix_map(&w->lo_narrow, wp_lo, kGateColumns, kp,
                                kProjectionNarrowWBoxRows)))
        return st;
    return LSTM_OK;
}

int launch_projection(const CUtensorMap &x_map, const ProjectionW &w, float *g, int rows, int kp,
                      int math, unsigned *fault, cudaStream_t stream, int *grid_out)
{
    if (math != LSTM_MATH_3XTF32 && math != LSTM_MATH_TF32)
        return fail(LSTM_E_INVALID, "projection: unknown math mode %d", math);
    if (rows <= 0)
        return fail(LSTM_E_INVALID, "projection: rows %d", rows);
    // G is written in 32 x 32 slices (one epilogue warp's rows), 128-byte swizzle
    CUtensorMap g_map;
    int st = encode_store_map(&g_map, g, rows, kGateColumns);
    if (st != LSTM_OK)
        return st;
    // few K blocks per tile: the W tile stays resident (see Shape)
    const bool resident = kp <= RESIDENT_KBLOCKS * BK;
    if (math == LSTM_MATH_TF32)
        return resident ? launch_tiles<GatesTf32ResidentShape>(x_map, w.hi, w.lo, g_map, rows, kp,
                                                                fault, stream, grid_out)
                        : launch_tiles<GatesTf32Shape>(x_map, w.hi, w.lo, g_map, rows, kp, fault,
                                                       stream, grid_out);
    // When the 256-column tiles would fill at most half of the CTAs that run
    // at once, 128-column tiles give every CTA half the work on twice as many
    // SMs.
    int dev = 0;
    if ((st = cuda_status(cudaGetDevice(&dev), "current device")))
        return st;
    const int fit = (dev >= 0 && dev < 64 && g_max_ctas[dev] > 0) ? g_max_ctas[dev] : 148;
    const long tiles = (static_cast<long>(rows) + BM - 1) / BM * GatesShape::TILES_N;
    if (2 * tiles <= fit)
        return resident ? launch_tiles<GatesNarrowResidentShape>(x_map, w.hi_narrow, w.lo_narrow,
                                                                 g_map, rows, kp, fault, stream, grid_out)
                        : launch_tiles<GatesNarrowShape>(x_map, w.hi_narrow, w.lo_narrow, g_map,
                                                         rows, kp, fault, stream, grid_out);
    return resident ? launch_tiles<GatesResidentShape>(x_map, w.hi, w.lo, g_map, rows, kp, fault,
                                                       stream, grid_out)
                    : launch_tiles<GatesShape>(x_map, w.hi, w.lo, g_map, rows, kp, fault, stream,
                                               grid_out);
}

} // namespace lstm
