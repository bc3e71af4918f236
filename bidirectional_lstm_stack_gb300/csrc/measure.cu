// Measurement entry points: the denominators the benchmark reports the
// kernels against, measured on the GPU it runs on.
//
// lstm_tf32_rate: the dense rate of the tensor cores in the mode the
// projection and the dense heads use (tcgen05.mma kind::tf32, M = 128,
// N = 256, fp32 accumulation in tensor memory).  One CTA per SM issues
// back-to-back MMAs from operands resident in shared memory into one
// accumulator, so nothing but the tensor pipe limits it.  The projection's
// 3xTF32 mode runs three such products per fp32 product; its roofline is a
// third of this rate.
#include <mutex>

#include "common.cuh"

namespace lstm {
namespace {

constexpr int RATE_THREADS = 128;
constexpr int RATE_M = 128, RATE_N = 256, RATE_K = 8;
constexpr int RATE_A_BYTES = RATE_M * 16 * 4;  // 128 rows x 16 fp32 (64-byte rows)
constexpr int RATE_B_BYTES = RATE_N * 16 * 4;  // 256 rows x 16 fp32
// Far more shared memory than the operands need, so that one CTA runs per
// SM and no two CTAs share a tensor pipe.
constexpr size_t RATE_SMEM = 160 * 1024;
constexpr uint64_t RATE_WAIT_NS = 2000000000ull;
constexpr uint32_t RATE_IDESC = ptx::tf32_idesc(RATE_M, RATE_N);

__global__ void __launch_bounds__(RATE_THREADS, 1)
tf32_rate_kernel(int iterations, unsigned *fault)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t done;
    __shared__ uint32_t tmem_slot;
    // operands: small TF32 values (exact), written by the generic proxy and
    // read by the tensor cores through the async proxy
    float *op = reinterpret_cast<float *>(smem);
    for (int i = threadIdx.x; i < (RATE_A_BYTES + RATE_B_BYTES) / 4; i += RATE_THREADS)
        op[i] = static_cast<float>(i % 7) * 0.25f - 0.75f;
    ptx::fence_proxy_async_smem();
    const int warp = threadIdx.x >> 5;
    if (warp == 0) {
        ptx::tmem_alloc(&tmem_slot, RATE_N);
        ptx::tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        ptx::mbar_init(&done, 1);
        ptx::fence_mbar_init();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t a = ptx::smem_u32(smem);
    const uint32_t b = a + RATE_A_BYTES;
    if (threadIdx.x == 0) {
        for (int it = 0; it < iterations; ++it) {
#pragma unroll
            for (int j = 0; j < 2; ++j)  // two K = 8 steps per 64-byte row
                ptx::mma_tf32(tmem, ptx::sw64_desc(a + j * 32), ptx::sw64_desc(b + j * 32),
                              RATE_IDESC, (it | j) != 0);
        }
        ptx::mma_commit(&done);
    }
    __syncwarp();
    if (warp == 0)
        ptx::mbar_wait_drain(&done, 0, fault, RATE_WAIT_NS);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 0)
        ptx::tmem_dealloc(tmem, RATE_N);
}

}  // namespace
}  // namespace lstm

using namespace lstm;

extern "C" int lstm_tf32_rate(int device, int iterations, double *tflops)
{
    if (!tflops)
        return fail(LSTM_E_INVALID, "lstm_tf32_rate: null output pointer");
    if (iterations <= 0 || iterations > 10000000)
        return fail(LSTM_E_INVALID, "lstm_tf32_rate: iterations %d outside 1..10^7", iterations);
    int st = prepare_device(device);
    if (st != LSTM_OK)
        return st;
    DeviceGuard guard(device);
    if (!guard.ok)
        return fail(LSTM_E_CUDA, "cannot make device %d current", device);
    int sms = 0;
    if ((st = cuda_status(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device),
                          "SM count")))
        return st;
    if ((st = cuda_status(cudaFuncSetAttribute(tf32_rate_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(RATE_SMEM)),
                          "rate kernel shared-memory attribute")))
        return st;
    unsigned *fault = fault_word();
    if (!fault)
        return fail(LSTM_E_CUDA, "cannot resolve the device fault word");
    cudaStream_t stream = nullptr;
    cudaEvent_t ev[2] = {};
    st = cuda_status(cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking), "rate stream");
    for (int i = 0; i < 2 && st == LSTM_OK; ++i)
        st = cuda_status(cudaEventCreate(&ev[i]), "rate event");
    float ms = 0.0f;
    unsigned bits = 0;
    if (st == LSTM_OK) {
        // a short warm-up launch, then the timed one
        const int warm = iterations / 10 > 0 ? iterations / 10 : 1;
        tf32_rate_kernel<<<sms, RATE_THREADS, RATE_SMEM, stream>>>(warm, fault);
        st = cuda_status(cudaGetLastError(), "rate kernel launch");
        if (st == LSTM_OK) st = cuda_status(cudaEventRecord(ev[0], stream), "event record");
        if (st == LSTM_OK) {
            tf32_rate_kernel<<<sms, RATE_THREADS, RATE_SMEM, stream>>>(iterations, fault);
            st = cuda_status(cudaGetLastError(), "rate kernel launch");
        }
        if (st == LSTM_OK) st = cuda_status(cudaEventRecord(ev[1], stream), "event record");
        if (st == LSTM_OK) st = cuda_status(cudaStreamSynchronize(stream), "rate kernel");
        if (st == LSTM_OK) st = cuda_status(cudaEventElapsedTime(&ms, ev[0], ev[1]), "elapsed");
        if (st == LSTM_OK)
            st = cuda_status(cudaMemcpy(&bits, fault, sizeof bits, cudaMemcpyDeviceToHost),
                             "fault word read");
    }
    for (cudaEvent_t e : ev)
        if (e)
            cudaEventDestroy(e);
    if (stream)
        cudaStreamDestroy(stream);
    if (st != LSTM_OK)
        return st;
    if (bits)
        return fail(LSTM_E_FAULT, "lstm_tf32_rate: a bounded wait ran out (fault bits 0x%x)", bits);
    const double flops = static_cast<double>(sms) * iterations * 2.0 /* K steps */ * 2.0 *
                         RATE_M * RATE_N * RATE_K;
    *tflops = flops / (static_cast<double>(ms) * 1e-3) / 1e12;
    return LSTM_OK;
}
