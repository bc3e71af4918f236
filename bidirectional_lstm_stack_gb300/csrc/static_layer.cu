// One bidirectional LSTM layer that allocates no device memory.
//
// Some callers cannot call cudaMalloc: code that runs while a CUDA graph is
// being captured (allocation is not a capturable operation), plug-ins whose
// host framework owns all device memory through its own arena and forbids
// allocations behind its back, and latency-critical loops where an
// allocation's implicit device synchronisation is not acceptable.  Those
// callers still pass their inputs, packed weights and outputs; the gate
// buffer the layer needs between its projection and its recurrences lives
// here in a fixed file-scope device array instead of a cudaMalloc'd one.
//
// The array holds kStaticRows rows of 1024 gate pre-activations (16 MiB).
// Every GPU that loads the library keeps it until the process exits.  All
// calls share it, so calls that overlap on the GPU (different streams, or
// different host threads) race on it and must be ordered by the caller.  It
// keeps the previous call's contents; nothing needs clearing, because each
// call's projection writes every row its recurrences then read.
#include <mutex>

#include "common.cuh"

namespace lstm {
namespace {

constexpr long kStaticRows = 4096;
__device__ __align__(256) float g_static_gates[kStaticRows * kGateColumns];

// Per-device set-up, with that device current: the kernels' per-device
// attributes (prepare_device) and the array's device address (a host-side
// name of a __device__ array is not a device address).
int static_setup(int device, float **gates)
{
    static std::mutex mu;
    static float *addr[64] = {};
    int st = prepare_device(device);  // also rejects devices out of range
    if (st != LSTM_OK)
        return st;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[device]) {
        void *p = nullptr;
        st = cuda_status(cudaGetSymbolAddress(&p, g_static_gates), "static gate buffer address");
        if (st != LSTM_OK)
            return st;
        addr[device] = static_cast<float *>(p);
    }
    *gates = addr[device];
    return LSTM_OK;
}

}  // namespace
}  // namespace lstm

using namespace lstm;

extern "C" int lstm_layer_forward_static(const float *x, int batch, int steps, int in_width,
                                         const float *wp_hi, const float *wp_lo, int kp,
                                         const float *rp, const float *bias, float *y,
                                         void *stream)
{
    if (!x || !wp_hi || !wp_lo || !rp || !bias || !y)
        return fail(LSTM_E_INVALID, "lstm_layer_forward_static: null pointer");
    if (batch <= 0 || steps <= 0)
        return fail(LSTM_E_INVALID, "lstm_layer_forward_static: batch %d, steps %d must be positive",
                    batch, steps);
    const long rows = static_cast<long>(batch) * steps;
    if (rows > kStaticRows)
        return fail(LSTM_E_INVALID,
                    "lstm_layer_forward_static: %d windows x %d steps = %ld rows exceed the static "
                    "gate buffer's %ld rows; use lstm_projection/lstm_recurrence with your own buffer",
                    batch, steps, rows, kStaticRows);
    if (in_width <= 0 || in_width > kp || kp % 32 != 0)
        return fail(LSTM_E_INVALID, "lstm_layer_forward_static: in_width %d, kp %d", in_width, kp);
    int st;
    if ((st = check_aligned(x, "static layer input")) || (st = check_aligned(wp_hi, "wp_hi")) ||
        (st = check_aligned(wp_lo, "wp_lo")) || (st = check_aligned(rp, "rp")) ||
        (st = check_aligned(bias, "bias")) || (st = check_aligned(y, "static layer output")))
        return st;
    int current = -1;
    if ((st = cuda_status(cudaGetDevice(&current), "current device")))
        return st;
    // every buffer lives on the current device, where the kernels run
    const struct {
        const void *p;
        const char *name;
    } buffers[] = {{x, "x"}, {wp_hi, "wp_hi"}, {wp_lo, "wp_lo"}, {rp, "rp"},
                   {bias, "bias"}, {y, "y"}};
    for (const auto &b : buffers) {
        int dev = -1;
        if ((st = pointer_device(b.p, &dev)))
            return st;
        if (dev != current)
            return fail(LSTM_E_INVALID,
                        "lstm_layer_forward_static: %s is on device %d, current device is %d",
                        b.name, dev, current);
    }
    float *gates = nullptr;
    if ((st = static_setup(current, &gates)) != LSTM_OK)
        return st;
    unsigned *fault = fault_word();
    if (!fault)
        return fail(LSTM_E_CUDA, "cannot resolve the device fault word");
    CUtensorMap xm;
    ProjectionW w;
    if ((st = encode_matrix_map(&xm, x, rows, in_width, kProjectionBoxRows)) ||
        (st = encode_projection_w(&w, wp_hi, wp_lo, kp)))
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = launch_projection(xm, w, gates, static_cast<int>(rows), kp, LSTM_MATH_3XTF32, fault,
                                s)))
        return st;
    return launch_recurrence(gates, rp, bias, y, batch, steps, kBothDirections, fault, s);
}
