// Input projection of one LSTM layer, both directions in one launch:
//     G[m][n] = sum_k X[m][k] * Wp[n][k],   m < rows, n < 1024,
// the dense `x . W^T` over every step of every window that the speakrs 0.6.0
// pages run per layer before the recurrence (lstmproj.rs module docs;
// `InputProjection::enqueue`), with the gate columns already in the packed,
// unit-interleaved order (the packer reorders W's rows).
//
// Design (sm_103a):
//  * one CTA computes a 128 x 256 tile of G; K advances in blocks of 32 fp32
//    (128 bytes, one 128-byte-swizzle row), double-buffered;
//  * a TMA producer warp loads the X block and the two TF32 planes of Wp
//    (hi and lo, split on the host) into 128B-swizzled shared memory;
//  * four converter warps split the X block in place into its TF32 hi part
//    and a second buffer with the TF32 lo remainder;
//  * one thread issues tcgen05.mma kind::tf32 (M=128, N=256, K=8) into a
//    tensor-memory accumulator: x_hi*w_hi + x_hi*w_lo + x_lo*w_hi, i.e. the
//    3xTF32 split that keeps fp32-level accuracy (the TF32 tensor fragments
//    of the pages' `spk_lstm_projection_tf32` were not accurate enough on
//    some parts, per `tf32_projection_accurate`);
//  * the converter warps then read the accumulator with tcgen05.ld and store
//    the rows of G.
// Every mbarrier wait is bounded in time; a wait that runs out sets a bit in
// the fault word and the CTA drains and returns.
#include <cudaTypedefs.h>
#include <mutex>

#include "common.cuh"

namespace lstm {
namespace {

constexpr int BM = 128;  // rows of G per CTA (MMA M)
constexpr int BN = 256;  // gate columns per CTA (MMA N)
constexpr int BK = 32;   // fp32 per K block = 128 bytes
constexpr int STAGES = 2;
constexpr int A_BYTES = BM * BK * 4;                     // 16 KiB
constexpr int B_BYTES = BN * BK * 4;                     // 32 KiB
constexpr int STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;   // A hi, A lo, B hi, B lo
constexpr uint32_t TX_BYTES = A_BYTES + 2 * B_BYTES;     // what TMA writes per stage
constexpr uint32_t TMEM_COLS = BN;                       // fp32 accumulator columns
constexpr int THREADS = 192;  // warps 0-3 convert + epilogue, 4 TMA, 5 MMA
constexpr int CONVERTERS = 128;
constexpr size_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s

// tcgen05 shared-memory matrix descriptor: K-major operand, 128-byte
// swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr)
{
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) |
           (static_cast<uint64_t>(1) << 16) |            // leading offset (unused, swizzled K-major)
           (static_cast<uint64_t>(1024 >> 4) << 32) |    // stride offset: 8 rows x 128 B
           (static_cast<uint64_t>(1) << 46) |            // descriptor version (tcgen05)
           (static_cast<uint64_t>(2) << 61);             // 128-byte swizzle
}

// Instruction descriptor, kind::tf32: D fp32, A and B TF32, both K-major,
// N = 256, M = 128.
constexpr uint32_t IDESC = (1u << 4) | (2u << 7) | (2u << 10) |
                           (static_cast<uint32_t>(BN >> 3) << 17) |
                           (static_cast<uint32_t>(BM >> 4) << 24);

__device__ __forceinline__ float tf32_rna(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

__device__ __forceinline__ void split4(float4 v, float4 &hi, float4 &lo)
{
    hi.x = tf32_rna(v.x); lo.x = tf32_rna(v.x - hi.x);
    hi.y = tf32_rna(v.y); lo.y = tf32_rna(v.y - hi.y);
    hi.z = tf32_rna(v.z); lo.z = tf32_rna(v.z - hi.z);
    hi.w = tf32_rna(v.w); lo.w = tf32_rna(v.w - hi.w);
}

// Waits without regard to the abort flag (used to drain in-flight work).
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity, unsigned *fault)
{
    if (ptx::mbar_try_wait(bar, parity))
        return;
    const uint64_t start = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer() - start > WAIT_LIMIT_NS) {
            atomicOr(fault, kFaultDrain);
            return;
        }
    }
}

__global__ void __launch_bounds__(THREADS, 1)
projection_kernel(const __grid_constant__ CUtensorMap x_map,
                  const __grid_constant__ CUtensorMap whi_map,
                  const __grid_constant__ CUtensorMap wlo_map, float *__restrict__ g, int rows,
                  int kblocks, unsigned *fault)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
    uint64_t *conv = full + STAGES;
    uint64_t *empty = conv + STAGES;
    uint64_t *acc_full = empty + STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN;
    const int m0 = blockIdx.y * BM;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&conv[s], CONVERTERS);
            ptx::mbar_init(&empty[s], 1);
        }
        ptx::mbar_init(acc_full, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 4 && lane == 0) {
        ptx::prefetch_tensormap(&x_map);
        ptx::prefetch_tensormap(&whi_map);
        ptx::prefetch_tensormap(&wlo_map);
    }
    if (warp == 5) {
        ptx::tmem_alloc(tmem_slot, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    int issued = 0;  // producer: K blocks whose loads were issued

    if (warp == 4) {
        if (lane == 0) {
            for (int kb = 0; kb < kblocks; ++kb) {
                const int s = kb % STAGES;
                const uint32_t n = kb / STAGES;
                if (n > 0 && !ptx::mbar_wait_bounded(&empty[s], (n - 1) & 1, abort_flag, fault,
                                                     kFaultProducer, WAIT_LIMIT_NS))
                    break;
                uint8_t *st = smem + s * STAGE_BYTES;
                ptx::mbar_arrive_expect_tx(&full[s], TX_BYTES);
                ptx::tma_load_2d(st, &x_map, &full[s], kb * BK, m0);
                ptx::tma_load_2d(st + 2 * A_BYTES, &whi_map, &full[s], kb * BK, n0);
                ptx::tma_load_2d(st + 2 * A_BYTES + B_BYTES, &wlo_map, &full[s], kb * BK, n0);
                issued = kb + 1;
            }
        }
    } else if (warp == 5) {
        if (lane == 0) {
            for (int kb = 0; kb < kblocks; ++kb) {
                const int s = kb % STAGES;
                const uint32_t n = kb / STAGES;
                if (!ptx::mbar_wait_bounded(&conv[s], n & 1, abort_flag, fault, kFaultMma,
                                            WAIT_LIMIT_NS))
                    break;
                ptx::tc_fence_after();
                const uint32_t a_hi = ptx::smem_u32(smem + s * STAGE_BYTES);
                const uint32_t a_lo = a_hi + A_BYTES;
                const uint32_t b_hi = a_hi + 2 * A_BYTES;
                const uint32_t b_lo = b_hi + B_BYTES;
#pragma unroll
                for (int j = 0; j < BK / 8; ++j) {
                    const uint32_t off = j * 32;  // 8 TF32 = 32 bytes along K
                    ptx::mma_tf32(tmem, sw128_desc(a_hi + off), sw128_desc(b_hi + off), IDESC,
                                  (kb | j) != 0);
                    ptx::mma_tf32(tmem, sw128_desc(a_hi + off), sw128_desc(b_lo + off), IDESC, 1);
                    ptx::mma_tf32(tmem, sw128_desc(a_lo + off), sw128_desc(b_hi + off), IDESC, 1);
                }
                ptx::mma_commit(&empty[s]);
            }
            ptx::mma_commit(acc_full);
        }
    } else {
        // warps 0-3: split X into TF32 hi/lo, then the epilogue
        const int tid = threadIdx.x;
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
            const int s = kb % STAGES;
            const uint32_t n = kb / STAGES;
            if (!ptx::mbar_wait_bounded(&full[s], n & 1, abort_flag, fault, kFaultConverter,
                                        WAIT_LIMIT_NS)) {
                ok = false;
                break;
            }
            float4 *a = reinterpret_cast<float4 *>(smem + s * STAGE_BYTES);
            float4 *alo = reinterpret_cast<float4 *>(smem + s * STAGE_BYTES + A_BYTES);
#pragma unroll
            for (int i = 0; i < A_BYTES / 16 / CONVERTERS; ++i) {
                const int idx = tid + i * CONVERTERS;
                float4 hi, lo;
                split4(a[idx], hi, lo);
                a[idx] = hi;
                alo[idx] = lo;
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&conv[s]);
        }
        bool got = ok && ptx::mbar_wait_bounded(acc_full, 0, abort_flag, fault, kFaultEpilogue,
                                                WAIT_LIMIT_NS);
        // tcgen05.ld is warp-collective: take the epilogue only if every lane may
        if (__all_sync(0xffffffffu, got)) {
            ptx::tc_fence_after();
            const int row = warp * 32 + lane;
            const long m = static_cast<long>(m0) + row;
            const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(tmem + lane_base + c * 32, r);
                ptx::tmem_ld_wait();
                if (m < rows) {
                    float4 *dst = reinterpret_cast<float4 *>(g + m * kGateColumns + n0 + c * 32);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        dst[q] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                             __uint_as_float(r[4 * q + 2]),
                                             __uint_as_float(r[4 * q + 3]));
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 4 && lane == 0) {
        // every issued TMA load has landed before the CTA's shared memory goes away
        for (int kb = issued - STAGES < 0 ? 0 : issued - STAGES; kb < issued; ++kb)
            drain_wait(&full[kb % STAGES], (kb / STAGES) & 1, fault);
    }
    if (warp == 5) {
        if (lane == 0)
            drain_wait(acc_full, 0, fault);  // every MMA has completed
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
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

} // namespace

int encode_matrix_map(CUtensorMap *map, const float *base, long rows, int cols, int box_rows)
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
    cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(LSTM_E_CUDA, "cuTensorMapEncodeTiled failed (%d) for %ld x %d", (int)r, rows,
                    cols);
    return LSTM_OK;
}

int projection_prepare(int)
{
    return cuda_status(cudaFuncSetAttribute(projection_kernel,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(SMEM_BYTES)),
                       "projection shared-memory attribute");
}

int launch_projection(const CUtensorMap &x_map, const CUtensorMap &whi_map,
                      const CUtensorMap &wlo_map, float *g, int rows, int kp, unsigned *fault,
                      cudaStream_t stream)
{
    if (rows <= 0 || kp <= 0 || kp % BK != 0)
        return fail(LSTM_E_INVALID, "projection: rows %d, kp %d", rows, kp);
    const long mtiles = (static_cast<long>(rows) + BM - 1) / BM;
    if (mtiles > 65535)
        return fail(LSTM_E_OVERFLOW, "projection: %d rows exceed %d", rows, 65535 * BM);
    dim3 grid(kGateColumns / BN, static_cast<unsigned>(mtiles));
    projection_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(x_map, whi_map, wlo_map, g, rows,
                                                             kp / BK, fault);
    return cuda_status(cudaGetLastError(), "projection launch");
}

} // namespace lstm
