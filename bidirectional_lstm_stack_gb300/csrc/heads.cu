// The dense heads of the segmentation model on the LSTM stack's output
// (speakrs 0.6.0 pages, segdense.rs: `Site::Linear0` a row-major 256-to-128
// projection `[k, n]` with bias and LeakyReLU, `Site::Linear1` 128-to-128 with
// bias and LeakyReLU, `Site::Linear2` 128-to-7 with bias and log-softmax;
// `DenseOxide`: those epilogues fused into the GEMMs), per row of y:
//     h1 = leaky(y W0 + b0),  h2 = leaky(h1 W1 + b1),
//     out = log_softmax(h2 W2 + b2)  (7 classes).
//
// Design (sm_103a): one persistent kernel, one CTA per SM, runs all three
// layers on 128-row tiles (each CTA loads its own W k-blocks; the 384 KiB of
// W planes stay in L2):
//  * warp 8 (TMA producer) streams, per tile, 16 k-blocks of y with W0 and
//    then 8 k-blocks of W1 through a 6-stage ring;
//  * warps 0-3 split the y blocks into TF32 hi (in place) and lo;
//  * one thread of warp 9 issues tcgen05.mma kind::tf32 (M = 128, N = 128):
//    linear0 as y_hi W0_hi + y_hi W0_lo + y_lo W0_hi into accumulator 1, then
//    linear1 with its A operand, h1 split into TF32 hi/lo, read straight from
//    tensor memory, into accumulator 2;
//  * warps 4-7 (epilogue; warp 4+q owns rows 32q..32q+31, one row per lane)
//    read accumulator 1, add b0, apply LeakyReLU, split h1 and write both
//    halves back into tensor memory for linear1; then read accumulator 2, add
//    b1, apply LeakyReLU and, still in registers, multiply h2 by the
//    classifier's 128 x 7 weights (fp32 FMAs whose weight operands come
//    straight from the constant bank: b0, b1, W2 and b2 are one kernel
//    parameter; a 16-column MMA would sit at its per-instruction floor), add
//    b2 and write the log-softmax of the 7 logits.
// Tensor memory (512 columns): accumulator 1 [0, 128), h1 hi [128, 256),
// h1 lo [256, 384), accumulator 2 [384, 512).  The MMA thread starts linear1
// of a tile once the epilogue has written its h1 (which also means it has
// read accumulator 1 and, before that, accumulator 2 of the previous tile);
// the epilogue rewrites h1 only after linear1 of the previous tile completed.
// Every wait is bounded in time; a wait that runs out sets a fault bit, every
// role stops, and the CTA drains its loads and MMAs before freeing tensor
// memory.
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <new>

#include "common.cuh"

using namespace lstm;

namespace {
constexpr int kIn = LSTM_STACK_OUTPUT;      // 256
constexpr int kMid = LSTM_HEADS_HIDDEN;     // 128
constexpr int kCls = LSTM_HEADS_CLASSES;    // 7
constexpr int kClsPad = 8;                  // classifier weight row, padded

constexpr int BM = 128;                     // rows per tile
constexpr int BK = 16;                      // fp32 per K block (64 bytes)
constexpr int K0_BLOCKS = kIn / BK;         // 16: linear0
constexpr int K1_BLOCKS = kMid / BK;        // 8: linear1
constexpr int BLOCKS_PER_TILE = K0_BLOCKS + K1_BLOCKS;
constexpr int A_BYTES = BM * BK * 4;        // 8 KiB
constexpr int W_BYTES = kMid * BK * 4;      // 8 KiB: one W k-block, 128 rows
constexpr int STAGE_BYTES = 2 * A_BYTES + 2 * W_BYTES;  // A hi, A lo, W hi, W lo
constexpr int A_LO = A_BYTES;
constexpr int W_HI = 2 * A_BYTES;
constexpr int W_LO = W_HI + W_BYTES;
constexpr int STAGES = 6;
constexpr int RING_BYTES = STAGES * STAGE_BYTES;  // 192 KiB
constexpr size_t SMEM_BYTES = RING_BYTES + 256 + 1024;

// The epilogues' parameters, passed by value as one kernel parameter (4.6
// KiB): with every index a compile-time constant (the epilogue loops are
// unrolled), each use is an operand read straight from the constant bank,
// with no load instruction.  From shared memory the classifier alone took
// two 128-bit loads per hidden unit and row, each costing four issue cycles
// though all lanes read the same address.
struct HeadsParams {
    float b0[kMid];
    float b1[kMid];
    float w2[kMid][kClsPad];  // row k: the 7 class weights of hidden unit k, padded
    float b2[kClsPad];
};
constexpr uint32_t ACC1 = 0, H1HI = 128, H1LO = 256, ACC2 = 384, TMEM_COLS = 512;
constexpr uint32_t IDESC = ptx::tf32_idesc(BM, kMid);
constexpr int CONVERTERS = 128;
constexpr int EPILOGUE = 128;
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int THREADS = 320;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
static_assert(kMid == kHeadWBoxRows, "W box rows");
static_assert(RING_BYTES % 1024 == 0 && STAGE_BYTES % 1024 == 0, "stage alignment");

__global__ void __launch_bounds__(THREADS, 1)
heads_kernel(const __grid_constant__ CUtensorMap y_map,
             const __grid_constant__ CUtensorMap w0hi_map,
             const __grid_constant__ CUtensorMap w0lo_map,
             const __grid_constant__ CUtensorMap w1hi_map,
             const __grid_constant__ CUtensorMap w1lo_map, const __grid_constant__ HeadsParams hp,
             float slope, float *__restrict__ logp, int rows, int tiles, unsigned *fault,
             unsigned long long wait_limit_ns, int withhold)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + RING_BYTES);
    uint64_t *conv = full + STAGES;
    uint64_t *empty = conv + STAGES;
    uint64_t *acc1_full = empty + STAGES;
    uint64_t *acc2_full = acc1_full + 1;
    uint64_t *ep1_done = acc2_full + 1;   // h1 in tensor memory (and accumulator 1 read)
    uint64_t *mma_done = ep1_done + 1;    // every MMA issued complete (teardown)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&conv[s], CONVERTERS);
            ptx::mbar_init(&empty[s], 1);  // the MMAs that read the stage completed
        }
        ptx::mbar_init(acc1_full, 1);
        ptx::mbar_init(acc2_full, 1);
        ptx::mbar_init(ep1_done, EPILOGUE);
        ptx::mbar_init(mma_done, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == PRODUCER_WARP && lane == 0) {
        ptx::prefetch_tensormap(&y_map);
        ptx::prefetch_tensormap(&w0hi_map);
        ptx::prefetch_tensormap(&w0lo_map);
        ptx::prefetch_tensormap(&w1hi_map);
        ptx::prefetch_tensormap(&w1lo_map);
    }
    if (warp == MMA_WARP) {
        ptx::tmem_alloc(tmem_slot, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int first = static_cast<int>(blockIdx.x);
    const int stride = static_cast<int>(gridDim.x);
    long issued = 0;  // producer: stages whose loads were issued

    if (warp == PRODUCER_WARP) {
        // failure test (`withhold`): nothing is loaded, so the converters'
        // waits run out
        if (lane == 0 && !withhold) {
            long kbi = 0;
            for (int t = first; t < tiles && !*abort_flag; t += stride) {
                const int m0 = t * BM;
                bool ok = true;
                for (int kb = 0; kb < BLOCKS_PER_TILE; ++kb, ++kbi) {
                    const int s = static_cast<int>(kbi % STAGES);
                    const uint32_t n = static_cast<uint32_t>(kbi / STAGES);
                    if (n > 0 && !ptx::mbar_wait_bounded(&empty[s], (n - 1) & 1, abort_flag, fault,
                                                         kFaultProducer, wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    uint8_t *st = smem + s * STAGE_BYTES;
                    if (kb < K0_BLOCKS) {
                        ptx::mbar_arrive_expect_tx(&full[s], A_BYTES + 2 * W_BYTES);
                        ptx::tma_load_2d(st, &y_map, &full[s], kb * BK, m0);
                        ptx::tma_load_2d(st + W_HI, &w0hi_map, &full[s], kb * BK, 0);
                        ptx::tma_load_2d(st + W_LO, &w0lo_map, &full[s], kb * BK, 0);
                    } else {
                        const int k = (kb - K0_BLOCKS) * BK;
                        ptx::mbar_arrive_expect_tx(&full[s], 2 * W_BYTES);
                        ptx::tma_load_2d(st + W_HI, &w1hi_map, &full[s], k, 0);
                        ptx::tma_load_2d(st + W_LO, &w1lo_map, &full[s], k, 0);
                    }
                    issued = kbi + 1;
                }
                if (!ok)
                    break;
            }
        }
    } else if (warp == MMA_WARP) {
        if (lane == 0) {
            long kbi = 0;
            int ti = 0;
            for (int t = first; t < tiles && !*abort_flag; t += stride, ++ti) {
                bool ok = true;
                // linear0 into accumulator 1 (the epilogue read it before it
                // wrote the previous tile's h1, which linear1 waited for)
                for (int kb = 0; kb < K0_BLOCKS && ok; ++kb, ++kbi) {
                    const int s = static_cast<int>(kbi % STAGES);
                    const uint32_t n = static_cast<uint32_t>(kbi / STAGES);
                    if (!ptx::mbar_wait_bounded(&conv[s], n & 1, abort_flag, fault, kFaultMma,
                                                wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a_hi = ptx::smem_u32(smem + s * STAGE_BYTES);
                    const uint32_t a_lo = a_hi + A_LO;
                    const uint32_t b_hi = a_hi + W_HI;
                    const uint32_t b_lo = a_hi + W_LO;
#pragma unroll
                    for (int j = 0; j < BK / 8; ++j) {
                        const uint32_t off = j * 32;  // 8 TF32 along K
                        ptx::mma_tf32(tmem + ACC1, ptx::sw64_desc(a_hi + off),
                                      ptx::sw64_desc(b_hi + off), IDESC, (kb | j) != 0);
                        ptx::mma_tf32(tmem + ACC1, ptx::sw64_desc(a_hi + off),
                                      ptx::sw64_desc(b_lo + off), IDESC, 1);
                        ptx::mma_tf32(tmem + ACC1, ptx::sw64_desc(a_lo + off),
                                      ptx::sw64_desc(b_hi + off), IDESC, 1);
                    }
                    ptx::mma_commit(&empty[s]);
                }
                ptx::mma_commit(acc1_full);  // also when stopping: frees the epilogue
                if (!ok)
                    break;
                // linear1 into accumulator 2 once h1 of this tile is in place
                if (!ptx::mbar_wait_bounded(ep1_done, ti & 1, abort_flag, fault, kFaultMma,
                                            wait_limit_ns))
                    break;
                ptx::tc_fence_after();
                for (int kb = 0; kb < K1_BLOCKS && ok; ++kb, ++kbi) {
                    const int s = static_cast<int>(kbi % STAGES);
                    const uint32_t n = static_cast<uint32_t>(kbi / STAGES);
                    if (!ptx::mbar_wait_bounded(&conv[s], n & 1, abort_flag, fault, kFaultMma,
                                                wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t b_hi = ptx::smem_u32(smem + s * STAGE_BYTES) + W_HI;
                    const uint32_t b_lo = b_hi + W_BYTES;
#pragma unroll
                    for (int j = 0; j < BK / 8; ++j) {
                        const uint32_t off = j * 32;
                        const uint32_t kcol = static_cast<uint32_t>(kb * BK + j * 8);
                        ptx::mma_tf32_tmem_a(tmem + ACC2, tmem + H1HI + kcol,
                                             ptx::sw64_desc(b_hi + off), IDESC, (kb | j) != 0);
                        ptx::mma_tf32_tmem_a(tmem + ACC2, tmem + H1HI + kcol,
                                             ptx::sw64_desc(b_lo + off), IDESC, 1);
                        ptx::mma_tf32_tmem_a(tmem + ACC2, tmem + H1LO + kcol,
                                             ptx::sw64_desc(b_hi + off), IDESC, 1);
                    }
                    ptx::mma_commit(&empty[s]);
                }
                ptx::mma_commit(acc2_full);
                if (!ok)
                    break;
            }
            // every MMA issued has completed before tensor memory is freed
            ptx::mma_commit(mma_done);
            ptx::mbar_wait_drain(mma_done, 0, fault, WAIT_LIMIT_NS);
        }
    } else if (warp < 4) {
        // converters: split the y blocks into TF32 hi (in place) and lo; the
        // W1 stages only pass through
        const int tid = threadIdx.x;
        long kbi = 0;
        for (int t = first; t < tiles && !*abort_flag; t += stride) {
            bool ok = true;
            for (int kb = 0; kb < BLOCKS_PER_TILE; ++kb, ++kbi) {
                const int s = static_cast<int>(kbi % STAGES);
                const uint32_t n = static_cast<uint32_t>(kbi / STAGES);
                if (!ptx::mbar_wait_bounded(&full[s], n & 1, abort_flag, fault, kFaultConverter,
                                            wait_limit_ns)) {
                    ok = false;
                    break;
                }
                if (kb < K0_BLOCKS) {
                    float4 *a = reinterpret_cast<float4 *>(smem + s * STAGE_BYTES);
                    float4 *alo = reinterpret_cast<float4 *>(smem + s * STAGE_BYTES + A_LO);
#pragma unroll
                    for (int i = 0; i < A_BYTES / 16 / CONVERTERS; ++i) {
                        const int idx = tid + i * CONVERTERS;
                        float4 hi, lo;
                        ptx::split4(a[idx], hi, lo);
                        a[idx] = hi;
                        alo[idx] = lo;
                    }
                    ptx::fence_proxy_async_smem();
                }
                ptx::mbar_arrive(&conv[s]);
            }
            if (!ok)
                break;
        }
    } else if (warp >= 4) {
        // epilogue: warp 4+q owns tensor-memory lanes (tile rows) 32q..32q+31
        const int q = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        int ti = 0;
        for (int t = first; t < tiles; t += stride, ++ti) {
            const long row = static_cast<long>(t) * BM + q * 32 + lane;
            bool got = ptx::mbar_wait_bounded(acc1_full, ti & 1, abort_flag, fault, kFaultEpilogue,
                                              wait_limit_ns);
            // tcgen05.ld / st are warp-collective: continue only if every lane may
            if (!__all_sync(0xffffffffu, got) || *abort_flag)
                break;
            ptx::tc_fence_after();
            // h1 = leaky(acc1 + b0), written back as TF32 hi/lo columns
#pragma unroll
            for (int c = 0; c < kMid / 32; ++c) {
                uint32_t r[32], hi[32], lo[32];
                ptx::tmem_ld_32x32b_x32(tmem + lane_base + ACC1 + c * 32, r);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    float v = __uint_as_float(r[j]) + hp.b0[c * 32 + j];
                    v = v >= 0.0f ? v : slope * v;
                    const float h = ptx::tf32_rna(v);
                    hi[j] = __float_as_uint(h);
                    lo[j] = __float_as_uint(ptx::tf32_rna(v - h));
                }
                ptx::tmem_st_32x32b_x32(tmem + lane_base + H1HI + c * 32, hi);
                ptx::tmem_st_32x32b_x32(tmem + lane_base + H1LO + c * 32, lo);
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(ep1_done);
            got = ptx::mbar_wait_bounded(acc2_full, ti & 1, abort_flag, fault, kFaultEpilogue,
                                         wait_limit_ns);
            if (!__all_sync(0xffffffffu, got) || *abort_flag)
                break;
            ptx::tc_fence_after();
            // h2 = leaky(acc2 + b1) in registers, z = h2 W2 + b2 (fp32 FMAs)
            float z[kClsPad];
#pragma unroll
            for (int j = 0; j < kClsPad; ++j)
                z[j] = 0.0f;
#pragma unroll
            for (int c = 0; c < kMid / 32; ++c) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(tmem + lane_base + ACC2 + c * 32, r);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    float v = __uint_as_float(r[k]) + hp.b1[c * 32 + k];
                    v = v >= 0.0f ? v : slope * v;
#pragma unroll
                    for (int j = 0; j < kCls; ++j)
                        z[j] = fmaf(v, hp.w2[c * 32 + k][j], z[j]);
                }
            }
            ptx::tc_fence_before();
            if (row < rows) {
                float zmax = -INFINITY;
#pragma unroll
                for (int j = 0; j < kCls; ++j) {
                    z[j] += hp.b2[j];
                    zmax = fmaxf(zmax, z[j]);
                }
                float sum = 0.0f;
#pragma unroll
                for (int j = 0; j < kCls; ++j)
                    sum += expf(z[j] - zmax);
                const float lse = zmax + logf(sum);
#pragma unroll
                for (int j = 0; j < kCls; ++j)
                    logp[row * kCls + j] = z[j] - lse;
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == PRODUCER_WARP && lane == 0) {
        // every issued TMA load has landed before the shared memory goes away
        for (long kb = issued - STAGES < 0 ? 0 : issued - STAGES; kb < issued; ++kb)
            ptx::mbar_wait_drain(&full[kb % STAGES], static_cast<uint32_t>(kb / STAGES) & 1, fault,
                                 WAIT_LIMIT_NS);
    }
    if (warp == MMA_WARP) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

int g_max_ctas[64] = {};

// Per-device set-up, with that device current: the kernel's shared-memory
// attribute and the number of its CTAs that run at once.
int heads_prepare(int device)
{
    static std::mutex mu;
    static bool done[64] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (done[device])
        return LSTM_OK;
    int st = cuda_status(cudaFuncSetAttribute(heads_kernel,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(SMEM_BYTES)),
                         "heads shared-memory attribute");
    if (st != LSTM_OK)
        return st;
    int sms = 0, per_sm = 0;
    st = cuda_status(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device),
                     "SM count");
    if (st != LSTM_OK)
        return st;
    st = cuda_status(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, heads_kernel, THREADS,
                                                                   SMEM_BYTES),
                     "heads occupancy");
    if (st != LSTM_OK)
        return st;
    g_max_ctas[device] = per_sm > 0 ? per_sm * sms : sms;
    done[device] = true;
    return LSTM_OK;
}
}  // namespace

struct lstm_heads {
    int device = 0;
    long max_rows = 0;
    float slope = 0.01f;
    float *weights = nullptr;  // one allocation: the packed W0 and W1 planes
    float *w0_hi = nullptr, *w0_lo = nullptr, *w1_hi = nullptr, *w1_lo = nullptr;
    HeadsParams params = {};   // b0, b1, W2 (rows padded to 8), b2: a kernel parameter
    CUtensorMap map_w0hi, map_w0lo, map_w1hi, map_w1lo;
    CUtensorMap map_y;
    const float *map_y_base = nullptr;
    long map_y_rows = -1;
    unsigned *fault = nullptr;
};

extern "C" void lstm_heads_destroy(lstm_heads *h)
{
    if (!h)
        return;
    DeviceGuard guard(h->device);
    cudaFree(h->weights);
    delete h;
}

extern "C" int lstm_heads_create(const float *w0, const float *b0, const float *w1,
                                 const float *b1, const float *w2, const float *b2,
                                 float negative_slope, int max_rows, int device,
                                 lstm_heads **out)
{
    if (!out)
        return fail(LSTM_E_INVALID, "lstm_heads_create: null output pointer");
    *out = nullptr;
    if (!w0 || !b0 || !w1 || !b1 || !w2 || !b2)
        return fail(LSTM_E_INVALID, "lstm_heads_create: null weight pointer");
    if (max_rows <= 0)
        return fail(LSTM_E_INVALID, "lstm_heads_create: max_rows %d", max_rows);
    int st = prepare_device(device);
    if (st != LSTM_OK)
        return st;
    DeviceGuard guard(device);
    if (!guard.ok)
        return fail(LSTM_E_CUDA, "cannot make device %d current", device);
    if ((st = heads_prepare(device)) != LSTM_OK)
        return st;
    lstm_heads *h = new (std::nothrow) lstm_heads();
    if (!h)
        return fail(LSTM_E_ALLOC, "lstm_heads_create: host allocation failed");
    h->device = device;
    h->max_rows = max_rows;
    h->slope = negative_slope;
    h->fault = fault_word();
    if (!h->fault) {
        lstm_heads_destroy(h);
        return fail(LSTM_E_CUDA, "cannot resolve the device fault word");
    }

    // W0 [256][128] and W1 [128][128] (row-major [k, n]) become K-major
    // [n][k] TF32 hi/lo planes; W2 [128][7] stays fp32, rows padded to 8, in
    // the kernel parameter with the biases
    const long n0 = static_cast<long>(kMid) * kIn, n1 = static_cast<long>(kMid) * kMid;
    const long o_w0hi = 0, o_w0lo = o_w0hi + n0, o_w1hi = o_w0lo + n0, o_w1lo = o_w1hi + n1;
    const long total = (o_w1lo + n1 + 63) / 64 * 64;
    float *host = static_cast<float *>(calloc(total, sizeof(float)));
    if (!host) {
        lstm_heads_destroy(h);
        return fail(LSTM_E_ALLOC, "lstm_heads_create: host staging allocation failed");
    }
    auto split = [](float v, float *hi, float *lo) {
        *hi = tf32_round(v);
        *lo = tf32_round(v - *hi);
    };
    for (int n = 0; n < kMid; ++n) {
        for (int k = 0; k < kIn; ++k)
            split(w0[static_cast<long>(k) * kMid + n], &host[o_w0hi + n * kIn + k],
                  &host[o_w0lo + n * kIn + k]);
        for (int k = 0; k < kMid; ++k)
            split(w1[static_cast<long>(k) * kMid + n], &host[o_w1hi + n * kMid + k],
                  &host[o_w1lo + n * kMid + k]);
        h->params.b0[n] = b0[n];
        h->params.b1[n] = b1[n];
    }
    for (int k = 0; k < kMid; ++k)
        for (int j = 0; j < kCls; ++j)
            h->params.w2[k][j] = w2[k * kCls + j];
    for (int j = 0; j < kCls; ++j)
        h->params.b2[j] = b2[j];
    cudaError_t e = device_alloc(reinterpret_cast<void **>(&h->weights), total * sizeof(float));
    if (e == cudaSuccess)
        e = cudaMemcpy(h->weights, host, total * sizeof(float), cudaMemcpyHostToDevice);
    free(host);
    if (e != cudaSuccess) {
        cudaGetLastError();
        lstm_heads_destroy(h);
        return fail(LSTM_E_ALLOC, "lstm_heads_create: device allocation: %s",
                    cudaGetErrorString(e));
    }
    h->w0_hi = h->weights + o_w0hi;
    h->w0_lo = h->weights + o_w0lo;
    h->w1_hi = h->weights + o_w1hi;
    h->w1_lo = h->weights + o_w1lo;
    if ((st = encode_matrix_map(&h->map_w0hi, h->w0_hi, kMid, kIn, kHeadWBoxRows)) ||
        (st = encode_matrix_map(&h->map_w0lo, h->w0_lo, kMid, kIn, kHeadWBoxRows)) ||
        (st = encode_matrix_map(&h->map_w1hi, h->w1_hi, kMid, kMid, kHeadWBoxRows)) ||
        (st = encode_matrix_map(&h->map_w1lo, h->w1_lo, kMid, kMid, kHeadWBoxRows))) {
        lstm_heads_destroy(h);
        return st;
    }
    *out = h;
    return LSTM_OK;
}

extern "C" int lstm_heads_forward(lstm_heads *h, const float *y, size_t y_len, float *logp,
                                  size_t logp_len, int rows, void *stream)
{
    if (!h || !y || !logp)
        return fail(LSTM_E_INVALID, "lstm_heads_forward: null pointer");
    if (rows <= 0 || rows > h->max_rows)
        return fail(LSTM_E_INVALID, "lstm_heads_forward: rows %d outside 1..%ld", rows,
                    h->max_rows);
    if (y_len != static_cast<size_t>(rows) * kIn)
        return fail(LSTM_E_LENGTH, "heads input: expected %zu floats, got %zu",
                    static_cast<size_t>(rows) * kIn, y_len);
    if (logp_len != static_cast<size_t>(rows) * kCls)
        return fail(LSTM_E_LENGTH, "heads output: expected %zu floats, got %zu",
                    static_cast<size_t>(rows) * kCls, logp_len);
    int st = check_aligned(y, "heads input");
    if (st != LSTM_OK)
        return st;
    if ((reinterpret_cast<uintptr_t>(logp) & 3) != 0)
        return fail(LSTM_E_INVALID, "heads output (%p) is not 4-byte aligned", (void *)logp);
    DeviceGuard guard(h->device);
    if (!guard.ok)
        return fail(LSTM_E_CUDA, "cannot make device %d current", h->device);
    int dy = -1, dp = -1;
    if ((st = pointer_device(y, &dy)) != LSTM_OK || (st = pointer_device(logp, &dp)) != LSTM_OK)
        return st;
    if (dy != h->device || dp != h->device)
        return fail(LSTM_E_INVALID, "heads buffers on devices %d/%d, heads object on %d", dy, dp,
                    h->device);
    if (y != h->map_y_base || rows != h->map_y_rows) {
        if ((st = encode_matrix_map(&h->map_y, y, rows, kIn, kProjectionBoxRows)) != LSTM_OK)
            return st;
        h->map_y_base = y;
        h->map_y_rows = rows;
    }
    const long tiles = (static_cast<long>(rows) + BM - 1) / BM;
    const int fit = g_max_ctas[h->device] > 0 ? g_max_ctas[h->device] : 148;
    const long grid = tiles < fit ? tiles : fit;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = static_cast<cudaStream_t>(stream);
    if ((st = check_launch_injection("heads launch")))
        return st;
    const int ntiles = static_cast<int>(tiles);
    const KernelTest test = kernel_test(kTestHeads);
    return cuda_status(cudaLaunchKernelEx(&cfg, heads_kernel, h->map_y, h->map_w0hi, h->map_w0lo,
                                          h->map_w1hi, h->map_w1lo,
                                          h->params, h->slope, logp,
                                          rows, ntiles, h->fault, test.wait_limit_ns,
                                          test.withhold),
                       "heads launch");
}
