// C ABI of liblstmstack.so: error reporting, the host weight packer, the
// stack object (create / forward / destroy) and the step-level entry points.
//
// The stack follows the plan/enqueue split of the speakrs 0.6.0 pages
// (lstmproj.rs `Oxide::with_recurrence` packs and uploads the four layers and
// allocates the gate buffer once; `Oxide::enqueue` checks lengths and runs,
// per layer, the projection and then both directions' recurrences, the
// reverse one on a side stream joined back before the next layer).  What
// differs: the projection runs once per layer for both directions (N = 1024),
// both directions' recurrences are one launch (their clusters alternate in
// one grid) on the caller's stream, so a forward is one chain of eight
// kernels instead of a fork and join per layer, each projection allowed to
// start while the recurrence before it ends (programmatic dependent
// launch); the layers
// ping-pong between two scratch buffers instead of overwriting the output in
// place; and there is no exchange buffer to clear (the recurrence exchanges h
// through distributed shared memory).
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <string>

#include "common.cuh"

namespace lstm {

namespace {
thread_local std::string g_last_error;
__device__ unsigned g_fault_word;
}  // namespace

int fail(int code, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

int cuda_status(cudaError_t err, const char *what)
{
    if (err == cudaSuccess)
        return LSTM_OK;
    return fail(LSTM_E_CUDA, "%s: %s (%s)", what, cudaGetErrorString(err), cudaGetErrorName(err));
}

namespace {
// Failure injection (lstm_test_* hooks): let `skip` calls through, then fail
// `count` of them.
struct Injection {
    std::mutex mu;
    int skip = 0;
    int count = 0;
    bool take()
    {
        std::lock_guard<std::mutex> lock(mu);
        if (count <= 0)
            return false;
        if (skip > 0) {
            --skip;
            return false;
        }
        --count;
        return true;
    }
    void set(int s, int c)
    {
        std::lock_guard<std::mutex> lock(mu);
        skip = s > 0 ? s : 0;
        count = c > 0 ? c : 0;
    }
};
Injection g_fail_allocs;
Injection g_fail_launches;
}  // namespace

cudaError_t device_alloc(void **p, size_t bytes)
{
    if (g_fail_allocs.take()) {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaMalloc(p, bytes);
}

int check_launch_injection(const char *what)
{
    if (g_fail_launches.take())
        return fail(LSTM_E_CUDA, "%s: injected launch failure (test hook)", what);
    return LSTM_OK;
}

namespace {
KernelTest g_kernel_test[kTestKernels][64];
}  // namespace

KernelTest kernel_test(int kernel)
{
    int dev = 0;
    if (kernel < 0 || kernel >= kTestKernels || cudaGetDevice(&dev) != cudaSuccess || dev < 0 ||
        dev >= 64)
        return KernelTest{};
    return g_kernel_test[kernel][dev];
}

int set_kernel_test(int kernel, int withhold, unsigned long long wait_limit_ns)
{
    int dev = 0;
    int st = cuda_status(cudaGetDevice(&dev), "current device");
    if (st != LSTM_OK)
        return st;
    if (kernel < 0 || kernel >= kTestKernels || dev < 0 || dev >= 64)
        return fail(LSTM_E_INVALID, "test setting: kernel %d, device %d out of range", kernel, dev);
    g_kernel_test[kernel][dev].wait_limit_ns = wait_limit_ns;
    g_kernel_test[kernel][dev].withhold = withhold;
    return LSTM_OK;
}

bool kernel_test_active(int device)
{
    if (device < 0 || device >= 64)
        return false;
    for (int k = 0; k < kTestKernels; ++k)
        if (g_kernel_test[k][device].withhold ||
            g_kernel_test[k][device].wait_limit_ns != kDefaultWaitLimitNs)
            return true;
    return false;
}

unsigned *fault_word()
{
    // one address per device; resolved with that device current
    static std::mutex mu;
    static unsigned *addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fault_word) != cudaSuccess)
            return nullptr;
        addr[dev] = static_cast<unsigned *>(p);
    }
    return addr[dev];
}

// Round-to-nearest (ties away from zero) to TF32: keep 10 mantissa bits.
float tf32_round(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    if ((u & 0x7f800000u) == 0x7f800000u)  // inf / nan: unchanged
        return x;
    u = (u + 0x1000u) & 0xffffe000u;
    float r;
    memcpy(&r, &u, 4);
    return r;
}

namespace {
int check_device(int device)
{
    cudaDeviceProp prop;
    int st = cuda_status(cudaGetDeviceProperties(&prop, device), "device properties");
    if (st != LSTM_OK)
        return st;
    if (prop.major != 10 || prop.minor != 3)
        return fail(LSTM_E_DEVICE, "device %d is compute capability %d.%d; the kernels are built for 10.3 (sm_103a)",
                    device, prop.major, prop.minor);
    int cluster = 0;
    st = cuda_status(cudaDeviceGetAttribute(&cluster, cudaDevAttrClusterLaunch, device),
                     "cluster-launch attribute");
    if (st != LSTM_OK)
        return st;
    if (!cluster)
        return fail(LSTM_E_DEVICE, "device %d does not support cluster launch", device);
    return LSTM_OK;
}
}  // namespace

int prepare_device(int device)
{
    static std::mutex mu;
    static bool done[64] = {};
    if (device < 0 || device >= 64)
        return fail(LSTM_E_INVALID, "device %d out of range", device);
    std::lock_guard<std::mutex> lock(mu);
    if (done[device])
        return LSTM_OK;
    DeviceGuard guard(device);  // occupancy queries below use the current device
    if (!guard.ok)
        return fail(LSTM_E_CUDA, "cannot make device %d current", device);
    int st = check_device(device);
    if (st == LSTM_OK)
        st = projection_prepare(device);
    if (st == LSTM_OK)
        st = recurrence_prepare(device);
    if (st == LSTM_OK)
        done[device] = true;
    return st;
}

int check_aligned(const void *p, const char *what)
{
    if ((reinterpret_cast<uintptr_t>(p) & 15) != 0)
        return fail(LSTM_E_INVALID, "%s (%p) is not 16-byte aligned", what, p);
    return LSTM_OK;
}

int pointer_device(const void *p, int *device)
{
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(LSTM_E_INVALID, "pointer %p is not known to CUDA", p);
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return fail(LSTM_E_INVALID, "pointer %p is not device memory", p);
    *device = attr.device;
    return LSTM_OK;
}

constexpr int kLayers = LSTM_STACK_LAYERS;
constexpr int kPhaseEvents = 3 * 2 * kLayers;  // (projection, fwd, rev) x (start, end) x layers

}  // namespace lstm

using namespace lstm;

struct lstm_stack {
    int device = 0;
    int max_batch = 0;
    int max_steps = 0;
    long max_rows = 0;
    int in_width[kLayers] = {};
    int kp[kLayers] = {};
    float *weights = nullptr;  // one allocation: all packed planes
    float *wp_hi[kLayers] = {};
    float *wp_lo[kLayers] = {};
    float *rp[kLayers] = {};
    float *bias[kLayers] = {};
    float *gates = nullptr;     // [max_rows][1024]
    float *ping[2] = {};        // [max_rows][256] each
    // Host-memory entry points: two staging slots, used in turn, so that one
    // call's output copy and the next call's input copy run while a forward
    // computes.  Input copies run on copy_in, output copies on copy_out;
    // per slot, `staged` marks its input copy done, `computed` its forward
    // done, `returned` its output copy done.
    float *x_stage[2] = {};     // [max_rows][60]
    float *y_stage[2] = {};     // [max_rows][256]
    cudaStream_t copy_in = nullptr;
    cudaStream_t copy_out = nullptr;
    cudaEvent_t staged[2] = {};
    cudaEvent_t computed[2] = {};
    cudaEvent_t returned[2] = {};
    int next_slot = 0;
    bool slot_pending[2] = {};  // enqueued since the last lstm_stack_host_sync
    ProjectionW map_w[kLayers];
    CUtensorMap map_ping[2];
    CUtensorMap map_x;
    const float *map_x_base = nullptr;
    long map_x_rows = -1;
    bool timing = false;
    bool timed_once = false;
    cudaEvent_t phase[kPhaseEvents] = {};
    unsigned *fault = nullptr;
    unsigned *fault_host = nullptr;  // pinned [2]: the fault word after each slot's forward
    // CUDA-graph replay of the forward pass, one instantiated graph per
    // argument set (least recently used evicted)
    struct Graph {
        const float *x = nullptr;
        float *y = nullptr;
        int batch = 0, steps = 0;
        bool timing = false;
        int math = LSTM_MATH_3XTF32;
        bool fused = false;
        cudaGraphExec_t exec = nullptr;
        unsigned long long used = 0;
    };
    static constexpr int kGraphs = 8;
    Graph graphs[kGraphs];
    unsigned long long uses = 0;
    bool use_graphs = true;
    cudaStream_t capture = nullptr;
    int math = LSTM_MATH_3XTF32;  // projection products
    int fused_max_batch = 0;      // batches up to this run the fused recurrence
    int fused_fit = -1;           // windows the device runs fused at once (-1: not queried)
};

extern "C" const char *lstm_stack_last_error(void)
{
    return g_last_error.c_str();
}

namespace {
// Source row block of gate k (k = 0..3 for i, f, g, o) in each gate order.
const int kGateBlocks[2][4] = {
    {0, 1, 2, 3},  // LSTM_GATES_IFGO: blocks i, f, g, o
    {0, 2, 3, 1},  // LSTM_GATES_IOFC: blocks i, o, f, c (ONNX)
};
}  // namespace

extern "C" int lstm_pack_layer(const float *w, const float *r, const float *b, int in_width,
                               int kp, float *wp_hi, float *wp_lo, float *rp, float *bias)
{
    return lstm_pack_layer_ordered(w, r, b, in_width, kp, LSTM_GATES_IFGO, wp_hi, wp_lo, rp,
                                   bias);
}

extern "C" int lstm_pack_layer_ordered(const float *w, const float *r, const float *b,
                                       int in_width, int kp, int gate_order, float *wp_hi,
                                       float *wp_lo, float *rp, float *bias)
{
    if (!w || !r || !b || !wp_hi || !wp_lo || !rp || !bias)
        return fail(LSTM_E_INVALID, "lstm_pack_layer: null pointer");
    if (gate_order != LSTM_GATES_IFGO && gate_order != LSTM_GATES_IOFC)
        return fail(LSTM_E_INVALID, "lstm_pack_layer: unknown gate order %d", gate_order);
    const int *block = kGateBlocks[gate_order];
    if (in_width <= 0 || kp < in_width || kp % 32 != 0)
        return fail(LSTM_E_INVALID, "lstm_pack_layer: in_width %d, kp %d (need 0 < in_width <= kp, kp %% 32 == 0)",
                    in_width, kp);
    const int H = kHidden;
    for (int d = 0; d < 2; ++d) {
        for (int u = 0; u < H; ++u) {
            for (int k = 0; k < 4; ++k) {
                const long src_row = static_cast<long>(d) * 4 * H + block[k] * H + u;
                const long dst_row = static_cast<long>(d) * 4 * H + 4 * u + k;  // interleaved
                for (int j = 0; j < kp; ++j) {
                    const float v = j < in_width ? w[src_row * in_width + j] : 0.0f;
                    const float hi = tf32_round(v);
                    wp_hi[dst_row * kp + j] = hi;
                    wp_lo[dst_row * kp + j] = tf32_round(v - hi);
                }
                for (int j = 0; j < H; ++j)
                    rp[dst_row * H + j] = r[src_row * H + j];
                const float *bd = b + static_cast<long>(d) * 8 * H;
                bias[static_cast<long>(d) * 4 * H + 4 * u + k] =
                    bd[block[k] * H + u] + bd[4 * H + block[k] * H + u];
            }
        }
    }
    return LSTM_OK;
}

extern "C" void lstm_stack_destroy(lstm_stack *s)
{
    if (!s)
        return;
    DeviceGuard guard(s->device);
    cudaDeviceSynchronize();
    cudaFree(s->weights);
    cudaFree(s->gates);
    cudaFree(s->ping[0]);
    cudaFree(s->ping[1]);
    for (int k = 0; k < 2; ++k) {
        cudaFree(s->x_stage[k]);
        cudaFree(s->y_stage[k]);
        for (cudaEvent_t e : {s->staged[k], s->computed[k], s->returned[k]})
            if (e)
                cudaEventDestroy(e);
    }
    if (s->fault_host)
        cudaFreeHost(s->fault_host);
    if (s->copy_in)
        cudaStreamDestroy(s->copy_in);
    if (s->copy_out)
        cudaStreamDestroy(s->copy_out);
    for (int i = 0; i < kPhaseEvents; ++i)
        if (s->phase[i])
            cudaEventDestroy(s->phase[i]);
    for (auto &gr : s->graphs)
        if (gr.exec)
            cudaGraphExecDestroy(gr.exec);
    if (s->capture)
        cudaStreamDestroy(s->capture);
    delete s;
}

extern "C" int lstm_stack_create(const lstm_stack_weights *weights, int max_batch, int max_steps,
                                 int device, lstm_stack **out)
{
    return lstm_stack_create_ordered(weights, LSTM_GATES_IFGO, max_batch, max_steps, device, out);
}

extern "C" int lstm_stack_create_ordered(const lstm_stack_weights *weights, int gate_order,
                                         int max_batch, int max_steps, int device,
                                         lstm_stack **out)
{
    if (!out)
        return fail(LSTM_E_INVALID, "lstm_stack_create: null output pointer");
    *out = nullptr;
    if (gate_order != LSTM_GATES_IFGO && gate_order != LSTM_GATES_IOFC)
        return fail(LSTM_E_INVALID, "lstm_stack_create: unknown gate order %d", gate_order);
    if (!weights)
        return fail(LSTM_E_INVALID, "lstm_stack_create: null weights");
    for (int l = 0; l < kLayers; ++l)
        if (!weights->w[l] || !weights->r[l] || !weights->b[l])
            return fail(LSTM_E_INVALID, "lstm_stack_create: layer %d has a null weight pointer", l);
    if (max_batch <= 0 || max_steps <= 0)
        return fail(LSTM_E_INVALID, "lstm_stack_create: max_batch %d, max_steps %d", max_batch,
                    max_steps);
    const long max_rows = static_cast<long>(max_batch) * max_steps;
    if (max_rows > 65535L * 128 || max_rows * kGateColumns > 0x7fffffffL * 4)
        return fail(LSTM_E_OVERFLOW, "lstm_stack_create: %ld rows exceed the kernels' indexing",
                    max_rows);
    int st = prepare_device(device);
    if (st != LSTM_OK)
        return st;
    DeviceGuard guard(device);
    if (!guard.ok)
        return fail(LSTM_E_CUDA, "cannot make device %d current", device);

    lstm_stack *s = new (std::nothrow) lstm_stack();
    if (!s)
        return fail(LSTM_E_ALLOC, "lstm_stack_create: host allocation failed");
    s->device = device;
    s->max_batch = max_batch;
    s->max_steps = max_steps;
    s->max_rows = max_rows;
    s->fault = fault_word();
    if (!s->fault) {
        lstm_stack_destroy(s);
        return fail(LSTM_E_CUDA, "cannot resolve the device fault word");
    }

    // pack on the host, then one upload
    long offs[kLayers][4];
    long total = 0;
    for (int l = 0; l < kLayers; ++l) {
        s->in_width[l] = l == 0 ? kFeatures : kOutput;
        s->kp[l] = (s->in_width[l] + 31) / 32 * 32;
        const long wsz = static_cast<long>(kGateColumns) * s->kp[l];
        offs[l][0] = total;  total += wsz;             // wp_hi
        offs[l][1] = total;  total += wsz;             // wp_lo
        offs[l][2] = total;  total += 2L * kGates * kHidden;  // rp
        offs[l][3] = total;  total += 2L * kGates;            // bias
        total = (total + 63) / 64 * 64;  // keep every plane 256-byte aligned
    }
    float *host = static_cast<float *>(calloc(total, sizeof(float)));
    if (!host) {
        lstm_stack_destroy(s);
        return fail(LSTM_E_ALLOC, "lstm_stack_create: host staging allocation failed");
    }
    for (int l = 0; l < kLayers; ++l) {
        st = lstm_pack_layer_ordered(weights->w[l], weights->r[l], weights->b[l], s->in_width[l],
                                     s->kp[l], gate_order, host + offs[l][0], host + offs[l][1],
                                     host + offs[l][2], host + offs[l][3]);
        if (st != LSTM_OK) {
            free(host);
            lstm_stack_destroy(s);
            return st;
        }
    }
    auto alloc = [&](float **p, long floats, const char *what) -> int {
        cudaError_t e = device_alloc(reinterpret_cast<void **>(p), floats * sizeof(float));
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(LSTM_E_ALLOC, "cudaMalloc of %s (%ld bytes): %s", what,
                        floats * static_cast<long>(sizeof(float)), cudaGetErrorString(e));
        }
        return LSTM_OK;
    };
    st = alloc(&s->weights, total, "packed weights");
    if (st == LSTM_OK)
        st = cuda_status(cudaMemcpy(s->weights, host, total * sizeof(float), cudaMemcpyHostToDevice),
                         "weight upload");
    free(host);
    if (st == LSTM_OK) st = alloc(&s->gates, max_rows * kGateColumns, "gate buffer");
    if (st == LSTM_OK) st = alloc(&s->ping[0], max_rows * kOutput, "layer buffer 0");
    if (st == LSTM_OK) st = alloc(&s->ping[1], max_rows * kOutput, "layer buffer 1");
    for (int k = 0; k < 2; ++k) {
        if (st == LSTM_OK) st = alloc(&s->x_stage[k], max_rows * kFeatures, "input staging");
        if (st == LSTM_OK) st = alloc(&s->y_stage[k], max_rows * kOutput, "output staging");
    }
    if (st == LSTM_OK)
        st = cuda_status(
            cudaMallocHost(reinterpret_cast<void **>(&s->fault_host), 2 * sizeof(unsigned)),
            "pinned fault words");
    if (st != LSTM_OK) {
        lstm_stack_destroy(s);
        return st;
    }
    for (int l = 0; l < kLayers && st == LSTM_OK; ++l) {
        s->wp_hi[l] = s->weights + offs[l][0];
        s->wp_lo[l] = s->weights + offs[l][1];
        s->rp[l] = s->weights + offs[l][2];
        s->bias[l] = s->weights + offs[l][3];
        st = encode_projection_w(&s->map_w[l], s->wp_hi[l], s->wp_lo[l], s->kp[l]);
    }
    for (int i = 0; i < 2 && st == LSTM_OK; ++i)
        st = encode_matrix_map(&s->map_ping[i], s->ping[i], max_rows, kOutput, kProjectionBoxRows);
    if (st == LSTM_OK)
        st = cuda_status(cudaStreamCreateWithFlags(&s->capture, cudaStreamNonBlocking),
                         "capture stream");
    if (st == LSTM_OK)
        st = cuda_status(cudaStreamCreateWithFlags(&s->copy_in, cudaStreamNonBlocking),
                         "input copy stream");
    if (st == LSTM_OK)
        st = cuda_status(cudaStreamCreateWithFlags(&s->copy_out, cudaStreamNonBlocking),
                         "output copy stream");
    for (int k = 0; k < 2 && st == LSTM_OK; ++k) {
        for (cudaEvent_t *e : {&s->staged[k], &s->computed[k], &s->returned[k]})
            if (st == LSTM_OK)
                st = cuda_status(cudaEventCreateWithFlags(e, cudaEventDisableTiming), "event");
    }
    for (int i = 0; i < kPhaseEvents && st == LSTM_OK; ++i)
        st = cuda_status(cudaEventCreate(&s->phase[i]), "phase event");
    if (st == LSTM_OK)
        st = cuda_status(cudaDeviceSynchronize(), "create");
    if (st != LSTM_OK) {
        lstm_stack_destroy(s);
        return st;
    }
    *out = s;
    return LSTM_OK;
}

namespace {

int check_forward_args(lstm_stack *s, const void *x, size_t x_len, const void *y, size_t y_len,
                       int batch, int steps)
{
    if (!s || !x || !y)
        return fail(LSTM_E_INVALID, "forward: null pointer");
    if (batch <= 0 || steps <= 0)
        return fail(LSTM_E_INVALID, "forward: batch %d, steps %d must be positive", batch, steps);
    if (batch > s->max_batch || steps > s->max_steps)
        return fail(LSTM_E_INVALID, "forward: batch %d x steps %d exceeds the created %d x %d",
                    batch, steps, s->max_batch, s->max_steps);
    const size_t rows = static_cast<size_t>(batch) * steps;
    if (x_len != rows * kFeatures)
        return fail(LSTM_E_LENGTH, "forward input: expected %zu floats, got %zu", rows * kFeatures,
                    x_len);
    if (y_len != rows * kOutput)
        return fail(LSTM_E_LENGTH, "forward output: expected %zu floats, got %zu", rows * kOutput,
                    y_len);
    return LSTM_OK;
}

// Whether a forward of `batch` windows runs the fused recurrence: enabled up
// to fused_max_batch, and only while both directions' clusters of one window
// each run at once on the device (larger batches take the projection kernel).
bool fused_batch(lstm_stack *s, int batch)
{
    if (batch > s->fused_max_batch)
        return false;
    if (s->fused_fit < 0) {
        int fit = -1;
        for (int kp : {64, 256}) {
            int n = 0;
            if (recurrence_fused_max_clusters(kp, &n) != LSTM_OK) {
                n = 0;
                cudaGetLastError();
            }
            fit = fit < 0 || n < fit ? n : fit;
        }
        s->fused_fit = fit / 2;
    }
    return batch <= s->fused_fit;
}

int forward_device(lstm_stack *s, const float *x, float *y, int batch, int steps,
                   cudaStream_t stream)
{
    const long rows = static_cast<long>(batch) * steps;
    int st;
    if (x != s->map_x_base || rows != s->map_x_rows) {
        st = encode_matrix_map(&s->map_x, x, rows, kFeatures, kProjectionBoxRows);
        if (st != LSTM_OK)
            return st;
        s->map_x_base = x;
        s->map_x_rows = rows;
    }
    // phase events: while the pass is being captured they are recorded as
    // external events, so they also fire when the graph is replayed (the flag
    // is valid only during capture; launched directly they are plain
    // records); the recurrence of both directions is one launch, so its time
    // fills both recurrence slots
    auto ev = [&](int layer, int part, int end) { return s->phase[(layer * 3 + part) * 2 + end]; };
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (s->timing && (st = cuda_status(cudaStreamIsCapturing(stream, &capture), "capture status")))
        return st;
    const unsigned record_flags =
        capture == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
    auto mark = [&](int layer, int part, int end) -> int {
        if (!s->timing)
            return LSTM_OK;
        return cuda_status(cudaEventRecordWithFlags(ev(layer, part, end), stream, record_flags),
                           "event");
    };
    const bool fused = fused_batch(s, batch);
    for (int l = 0; l < kLayers; ++l) {
        const CUtensorMap &src = l == 0 ? s->map_x : s->map_ping[(l - 1) & 1];
        float *dst = l == kLayers - 1 ? y : s->ping[l & 1];
        if (fused) {
            // the projection computed inside the recurrence (an empty
            // projection phase)
            const float *xin = l == 0 ? x : s->ping[(l - 1) & 1];
            if ((st = mark(l, 0, 0)) || (st = mark(l, 0, 1)) || (st = mark(l, 1, 0)) ||
                (st = mark(l, 2, 0)))
                return st;
            if ((st = launch_recurrence_fused(xin, s->in_width[l], s->wp_hi[l], s->wp_lo[l],
                                              s->kp[l], s->rp[l], s->bias[l], dst, batch, steps,
                                              kBothDirections, s->fault, stream)))
                return st;
            if ((st = mark(l, 1, 1)) || (st = mark(l, 2, 1)))
                return st;
            continue;
        }
        if ((st = mark(l, 0, 0)))
            return st;
        int proj_ctas = 0;
        st = launch_projection(src, s->map_w[l], s->gates, static_cast<int>(rows), s->kp[l],
                               s->math, s->fault, stream, &proj_ctas);
        if (st != LSTM_OK)
            return st;
        if ((st = mark(l, 0, 1)) || (st = mark(l, 1, 0)) || (st = mark(l, 2, 0)))
            return st;
        // forward and reverse in one grid on the caller's stream: the next
        // layer's projection follows it on the same stream; with few windows
        // (both grids fit on the SMs side by side) it starts while the
        // projection runs (phase timing puts an event between them, so
        // there it starts after)
        if ((st = launch_recurrence(s->gates, s->rp[l], s->bias[l], dst, batch, steps,
                                    kBothDirections, s->fault, stream,
                                    s->timing ? -1 : proj_ctas)))
            return st;
        if ((st = mark(l, 1, 1)) || (st = mark(l, 2, 1)))
            return st;
    }
    if (s->timing)
        s->timed_once = true;
    return LSTM_OK;
}

}  // namespace

namespace {

// Runs the forward pass on `stream` by replaying a CUDA graph of it: the
// first call with a given (x, y, batch, steps, timing, math) records the launches
// on a private stream and instantiates the graph;
// later calls only launch it.  When `stream` is itself being captured (the
// caller is building a graph) or replay is off, the launches are enqueued
// directly.
int forward_replay(lstm_stack *s, const float *x, float *y, int batch, int steps,
                   cudaStream_t stream)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    int st = cuda_status(cudaStreamIsCapturing(stream, &cs), "stream capture status");
    if (st != LSTM_OK)
        return st;
    if (!s->use_graphs || cs != cudaStreamCaptureStatusNone || kernel_test_active(s->device))
        return forward_device(s, x, y, batch, steps, stream);
    lstm_stack::Graph *hit = nullptr, *victim = &s->graphs[0];
    for (auto &gr : s->graphs) {
        if (gr.exec && gr.x == x && gr.y == y && gr.batch == batch && gr.steps == steps &&
            gr.timing == s->timing && gr.math == s->math && gr.fused == fused_batch(s, batch)) {
            hit = &gr;
            break;
        }
        if (!gr.exec || (victim->exec && gr.used < victim->used))
            victim = &gr;
    }
    if (!hit) {
        if (victim->exec) {
            cudaGraphExecDestroy(victim->exec);
            victim->exec = nullptr;
        }
        st = cuda_status(cudaStreamBeginCapture(s->capture, cudaStreamCaptureModeThreadLocal),
                         "begin capture");
        if (st != LSTM_OK)
            return st;
        const int fst = forward_device(s, x, y, batch, steps, s->capture);
        cudaGraph_t graph = nullptr;
        st = cuda_status(cudaStreamEndCapture(s->capture, &graph), "end capture");
        if (fst != LSTM_OK || st != LSTM_OK) {
            if (graph)
                cudaGraphDestroy(graph);
            return fst != LSTM_OK ? fst : st;
        }
        cudaGraphExec_t exec = nullptr;
        st = cuda_status(cudaGraphInstantiate(&exec, graph, 0), "graph instantiate");
        cudaGraphDestroy(graph);
        if (st != LSTM_OK)
            return st;
        *victim = lstm_stack::Graph{x,         y,
                                    batch,     steps,
                                    s->timing, s->math,
                                    fused_batch(s, batch), exec,
                                    0};
        hit = victim;
    }
    hit->used = ++s->uses;
    if ((st = cuda_status(cudaGraphLaunch(hit->exec, stream), "graph launch")))
        return st;
    // a graph captured with phase timing records the phase events on replay
    if (s->timing)
        s->timed_once = true;
    return LSTM_OK;
}

}  // namespace

extern "C" int lstm_stack_set_graphs(lstm_stack *s, int enable)
{
    if (!s)
        return fail(LSTM_E_INVALID, "set_graphs: null stack");
    s->use_graphs = enable != 0;
    return LSTM_OK;
}

extern "C" int lstm_stack_set_math(lstm_stack *s, int math)
{
    if (!s)
        return fail(LSTM_E_INVALID, "set_math: null stack");
    if (math != LSTM_MATH_3XTF32 && math != LSTM_MATH_TF32)
        return fail(LSTM_E_INVALID, "set_math: unknown math mode %d", math);
    s->math = math;
    return LSTM_OK;
}

extern "C" int lstm_stack_set_fused_batches(lstm_stack *s, int max_batch)
{
    if (!s)
        return fail(LSTM_E_INVALID, "set_fused_batches: null stack");
    if (max_batch < 0)
        return fail(LSTM_E_INVALID, "set_fused_batches: max_batch %d", max_batch);
    s->fused_max_batch = max_batch;
    return LSTM_OK;
}

extern "C" int lstm_stack_forward(lstm_stack *s, const float *x, size_t x_len, float *y,
                                  size_t y_len, int batch, int steps, void *stream)
{
    int st = check_forward_args(s, x, x_len, y, y_len, batch, steps);
    if (st != LSTM_OK)
        return st;
    if ((st = check_aligned(x, "forward input")) != LSTM_OK)
        return st;
    if ((st = check_aligned(y, "forward output")) != LSTM_OK)
        return st;
    DeviceGuard guard(s->device);
    if (!guard.ok)
        return fail(LSTM_E_CUDA, "cannot make device %d current", s->device);
    int dx = -1, dy = -1;
    if ((st = pointer_device(x, &dx)) != LSTM_OK || (st = pointer_device(y, &dy)) != LSTM_OK)
        return st;
    if (dx != s->device || dy != s->device)
        return fail(LSTM_E_INVALID, "forward: buffers on devices %d/%d, stack on device %d", dx, dy,
                    s->device);
    return forward_replay(s, x, y, batch, steps, static_cast<cudaStream_t>(stream));
}

extern "C" int lstm_stack_forward_host_async(lstm_stack *s, const float *x_host, size_t x_len,
                                             float *y_host, size_t y_len, int batch, int steps,
                                             void *stream)
{
    int st = check_forward_args(s, x_host, x_len, y_host, y_len, batch, steps);
    if (st != LSTM_OK)
        return st;
    DeviceGuard guard(s->device);
    if (!guard.ok)
        return fail(LSTM_E_CUDA, "cannot make device %d current", s->device);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
    if ((st = cuda_status(cudaStreamIsCapturing(cs, &capturing), "capture status")))
        return st;
    if (capturing != cudaStreamCaptureStatusNone)
        return fail(LSTM_E_INVALID,
                    "forward_host_async: the stream is being captured (use lstm_stack_forward)");
    const int k = s->next_slot;
    // input: into slot k once the forward that last read it is done
    if ((st = cuda_status(cudaStreamWaitEvent(s->copy_in, s->computed[k]), "event wait")) ||
        (st = cuda_status(cudaMemcpyAsync(s->x_stage[k], x_host, x_len * sizeof(float),
                                          cudaMemcpyHostToDevice, s->copy_in),
                          "input copy")) ||
        (st = cuda_status(cudaEventRecord(s->staged[k], s->copy_in), "event record")))
        return st;
    // the forward: after its input copy, after the output copy that last read
    // slot k, and after the other slot's forward (the scratch is shared)
    if ((st = cuda_status(cudaStreamWaitEvent(cs, s->staged[k]), "event wait")) ||
        (st = cuda_status(cudaStreamWaitEvent(cs, s->returned[k]), "event wait")) ||
        (st = cuda_status(cudaStreamWaitEvent(cs, s->computed[k ^ 1]), "event wait")))
        return st;
    if ((st = forward_replay(s, s->x_stage[k], s->y_stage[k], batch, steps, cs)))
        return st;
    if ((st = cuda_status(cudaEventRecord(s->computed[k], cs), "event record")))
        return st;
    // output, and the kernels' fault word with it
    if ((st = cuda_status(cudaStreamWaitEvent(s->copy_out, s->computed[k]), "event wait")) ||
        (st = cuda_status(cudaMemcpyAsync(y_host, s->y_stage[k], y_len * sizeof(float),
                                          cudaMemcpyDeviceToHost, s->copy_out),
                          "output copy")) ||
        (st = cuda_status(cudaMemcpyAsync(&s->fault_host[k], s->fault, sizeof(unsigned),
                                          cudaMemcpyDeviceToHost, s->copy_out),
                          "fault word copy")) ||
        (st = cuda_status(cudaEventRecord(s->returned[k], s->copy_out), "event record")))
        return st;
    s->slot_pending[k] = true;
    s->next_slot = k ^ 1;
    return LSTM_OK;
}

extern "C" int lstm_stack_host_sync(lstm_stack *s)
{
    if (!s)
        return fail(LSTM_E_INVALID, "host_sync: null stack");
    DeviceGuard guard(s->device);
    if (!guard.ok)
        return fail(LSTM_E_CUDA, "cannot make device %d current", s->device);
    int st = cuda_status(cudaStreamSynchronize(s->copy_out), "output copies");
    if (st == LSTM_OK)
        st = cuda_status(cudaStreamSynchronize(s->copy_in), "input copies");
    if (st != LSTM_OK)
        return st;
    unsigned bits = 0;
    for (int k = 0; k < 2; ++k) {
        if (s->slot_pending[k])
            bits |= s->fault_host[k];
        s->slot_pending[k] = false;
    }
    if (bits) {
        cudaMemset(s->fault, 0, sizeof(unsigned));
        return fail(LSTM_E_FAULT,
                    "forward_host: a kernel's bounded wait ran out (fault bits 0x%x); the "
                    "result is not valid",
                    bits);
    }
    return LSTM_OK;
}

extern "C" int lstm_stack_forward_host(lstm_stack *s, const float *x_host, size_t x_len,
                                       float *y_host, size_t y_len, int batch, int steps,
                                       void *stream)
{
    const int st = lstm_stack_forward_host_async(s, x_host, x_len, y_host, y_len, batch, steps,
                                                 stream);
    if (st != LSTM_OK)
        return st;
    return lstm_stack_host_sync(s);
}

extern "C" int lstm_stack_enable_phase_timing(lstm_stack *s, int enable)
{
    if (!s)
        return fail(LSTM_E_INVALID, "enable_phase_timing: null stack");
    s->timing = enable != 0;
    s->timed_once = false;
    return LSTM_OK;
}

extern "C" int lstm_stack_phase_times(lstm_stack *s, float *ms)
{
    if (!s || !ms)
        return fail(LSTM_E_INVALID, "phase_times: null pointer");
    if (!s->timed_once)
        return fail(LSTM_E_INVALID, "phase_times: no timed forward since timing was enabled");
    DeviceGuard guard(s->device);
    for (int i = 0; i < 3 * kLayers; ++i) {
        int st = cuda_status(cudaEventSynchronize(s->phase[2 * i + 1]), "phase event sync");
        if (st == LSTM_OK)
            st = cuda_status(cudaEventElapsedTime(&ms[i], s->phase[2 * i], s->phase[2 * i + 1]),
                             "phase elapsed");
        if (st != LSTM_OK)
            return st;
    }
    return LSTM_OK;
}

extern "C" int lstm_projection(const float *x, int rows, int in_width, const float *wp_hi,
                               const float *wp_lo, int kp, float *g, void *stream)
{
    return lstm_projection_math(x, rows, in_width, wp_hi, wp_lo, kp, g, LSTM_MATH_3XTF32, stream);
}

extern "C" int lstm_projection_math(const float *x, int rows, int in_width, const float *wp_hi,
                                    const float *wp_lo, int kp, float *g, int math, void *stream)
{
    if (math != LSTM_MATH_3XTF32 && math != LSTM_MATH_TF32)
        return fail(LSTM_E_INVALID, "lstm_projection: unknown math mode %d", math);
    // the single-product mode never reads the lo plane
    if (math == LSTM_MATH_TF32 && !wp_lo)
        wp_lo = wp_hi;
    if (!x || !wp_hi || !wp_lo || !g)
        return fail(LSTM_E_INVALID, "lstm_projection: null pointer");
    if (rows <= 0 || in_width <= 0 || in_width > kp || kp % 32 != 0)
        return fail(LSTM_E_INVALID, "lstm_projection: rows %d, in_width %d, kp %d", rows, in_width,
                    kp);
    int st;
    if ((st = check_aligned(x, "projection input")) || (st = check_aligned(wp_hi, "wp_hi")) ||
        (st = check_aligned(wp_lo, "wp_lo")) || (st = check_aligned(g, "projection output")))
        return st;
    int dev = 0;
    if ((st = pointer_device(x, &dev)))
        return st;
    if ((st = prepare_device(dev)))
        return st;
    DeviceGuard guard(dev);
    unsigned *fault = fault_word();
    if (!fault)
        return fail(LSTM_E_CUDA, "cannot resolve the device fault word");
    CUtensorMap xm;
    ProjectionW w;
    if ((st = encode_matrix_map(&xm, x, rows, in_width, kProjectionBoxRows)) ||
        (st = encode_projection_w(&w, wp_hi, wp_lo, kp)))
        return st;
    return launch_projection(xm, w, g, rows, kp, math, fault, static_cast<cudaStream_t>(stream));
}

namespace {
int recurrence_args(const float *g, const float *rp, const float *bias, float *y, int batch,
                    int steps, int direction, int *dev)
{
    if (!g || !rp || !bias || !y)
        return fail(LSTM_E_INVALID, "lstm_recurrence: null pointer");
    if (batch <= 0 || steps <= 0)
        return fail(LSTM_E_INVALID, "lstm_recurrence: batch %d, steps %d", batch, steps);
    if (direction != 0 && direction != 1 && direction != LSTM_BOTH_DIRECTIONS)
        return fail(LSTM_E_INVALID,
                    "lstm_recurrence: direction %d (0 forward, 1 reverse, %d both)", direction,
                    LSTM_BOTH_DIRECTIONS);
    if (static_cast<long>(batch) * steps > 65535L * 128)
        return fail(LSTM_E_OVERFLOW, "lstm_recurrence: %d x %d rows exceed %ld", batch, steps,
                    65535L * 128);
    int st;
    if ((st = check_aligned(g, "g")) || (st = check_aligned(rp, "rp")) ||
        (st = check_aligned(y, "y")) || (st = pointer_device(g, dev)))
        return st;
    return prepare_device(*dev);
}

// The public direction (0, 1, LSTM_BOTH_DIRECTIONS) as the launchers take it.
int launch_direction(int direction)
{
    return direction == LSTM_BOTH_DIRECTIONS ? kBothDirections : direction;
}
}  // namespace

extern "C" int lstm_recurrence(const float *g, const float *rp, const float *bias, float *y,
                               int batch, int steps, int direction, void *stream)
{
    int dev = 0;
    int st = recurrence_args(g, rp, bias, y, batch, steps, direction, &dev);
    if (st != LSTM_OK)
        return st;
    DeviceGuard guard(dev);
    unsigned *fault = fault_word();
    if (!fault)
        return fail(LSTM_E_CUDA, "cannot resolve the device fault word");
    return launch_recurrence(g, rp, bias, y, batch, steps, launch_direction(direction), fault,
                             static_cast<cudaStream_t>(stream));
}

extern "C" int lstm_recurrence_floor(const float *g, const float *rp, const float *bias, float *y,
                                     int batch, int steps, int direction, void *stream)
{
    int dev = 0;
    int st = recurrence_args(g, rp, bias, y, batch, steps, direction, &dev);
    if (st != LSTM_OK)
        return st;
    DeviceGuard guard(dev);
    unsigned *fault = fault_word();
    if (!fault)
        return fail(LSTM_E_CUDA, "cannot resolve the device fault word");
    return launch_recurrence_floor(g, rp, bias, y, batch, steps, launch_direction(direction), fault,
                                   static_cast<cudaStream_t>(stream));
}

extern "C" int lstm_recurrence_fused(const float *x, int in_width, const float *wp_hi,
                                     const float *wp_lo, int kp, const float *rp,
                                     const float *bias, float *y, int batch, int steps,
                                     int direction, void *stream)
{
    if (!x || !wp_hi || !wp_lo)
        return fail(LSTM_E_INVALID, "lstm_recurrence_fused: null pointer");
    int dev = 0;
    // the argument checks of lstm_recurrence, with x standing in for G
    int st = recurrence_args(x, rp, bias, y, batch, steps, direction, &dev);
    if (st != LSTM_OK)
        return st;
    if ((st = check_aligned(wp_hi, "wp_hi")) || (st = check_aligned(wp_lo, "wp_lo")))
        return st;
    DeviceGuard guard(dev);
    int fit = 0;
    if ((st = recurrence_fused_max_clusters(kp, &fit)))
        return st;
    const long clusters = static_cast<long>(batch) * (direction == LSTM_BOTH_DIRECTIONS ? 2 : 1);
    if (clusters > fit)
        return fail(LSTM_E_INVALID,
                    "lstm_recurrence_fused: %ld clusters of one window each, the device runs %d "
                    "at once",
                    clusters, fit);
    unsigned *fault = fault_word();
    if (!fault)
        return fail(LSTM_E_CUDA, "cannot resolve the device fault word");
    return launch_recurrence_fused(x, in_width, wp_hi, wp_lo, kp, rp, bias, y, batch, steps,
                                   launch_direction(direction), fault,
                                   static_cast<cudaStream_t>(stream));
}

extern "C" int lstm_recurrence_variant(const float *g, const float *rp, const float *bias,
                                       float *y, int batch, int steps, int direction,
                                       int cluster_size, int windows_per_chunk, int chunks,
                                       int threads_per_block, void *stream)
{
    int dev = 0;
    int st = recurrence_args(g, rp, bias, y, batch, steps, direction, &dev);
    if (st != LSTM_OK)
        return st;
    DeviceGuard guard(dev);
    unsigned *fault = fault_word();
    if (!fault)
        return fail(LSTM_E_CUDA, "cannot resolve the device fault word");
    return launch_recurrence_variant(g, rp, bias, y, batch, steps, launch_direction(direction), cluster_size,
                                     windows_per_chunk, chunks, threads_per_block, fault,
                                     static_cast<cudaStream_t>(stream));
}

extern "C" int lstm_recurrence_max_clusters(int cluster_size, int windows_per_chunk, int chunks,
                                            int threads_per_block, int device,
                                            int *max_clusters)
{
    if (!max_clusters)
        return fail(LSTM_E_INVALID, "lstm_recurrence_max_clusters: null pointer");
    int st = prepare_device(device);
    if (st != LSTM_OK)
        return st;
    DeviceGuard guard(device);
    return recurrence_max_clusters(cluster_size, windows_per_chunk, chunks, threads_per_block,
                                   max_clusters);
}

extern "C" int lstm_fault_status(unsigned int *fault)
{
    if (!fault)
        return fail(LSTM_E_INVALID, "lstm_fault_status: null pointer");
    int st = cuda_status(cudaDeviceSynchronize(), "fault status synchronize");
    if (st != LSTM_OK)
        return st;
    unsigned zero = 0;
    if ((st = cuda_status(cudaMemcpyFromSymbol(fault, g_fault_word, sizeof(unsigned)),
                          "fault word read")))
        return st;
    return cuda_status(cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(unsigned)), "fault word clear");
}

// ---- failure-injection hooks (tests only) ----------------------------------

extern "C" int lstm_test_fail_allocations(int skip, int count)
{
    g_fail_allocs.set(skip, count);
    return LSTM_OK;
}

extern "C" int lstm_test_fail_launches(int skip, int count)
{
    g_fail_launches.set(skip, count);
    return LSTM_OK;
}

namespace {
int set_timeout_test(int kernel, const char *what, int withhold, unsigned int wait_limit_us,
                     int device)
{
    if (wait_limit_us > 2000000u)
        return fail(LSTM_E_INVALID, "%s test: wait limit %u us above 2 s", what, wait_limit_us);
    int st = prepare_device(device);
    if (st != LSTM_OK)
        return st;
    DeviceGuard guard(device);
    if (!guard.ok)
        return fail(LSTM_E_CUDA, "cannot make device %d current", device);
    const unsigned long long limit =
        wait_limit_us ? wait_limit_us * 1000ull : kDefaultWaitLimitNs;  // 0: the default 2 s
    return set_kernel_test(kernel, withhold != 0, limit);
}
}  // namespace

extern "C" int lstm_test_recurrence_timeout(int withhold, unsigned int wait_limit_us, int device)
{
    return set_timeout_test(kTestRecurrence, "recurrence", withhold, wait_limit_us, device);
}

extern "C" int lstm_test_projection_timeout(int withhold, unsigned int wait_limit_us, int device)
{
    return set_timeout_test(kTestProjection, "projection", withhold, wait_limit_us, device);
}

extern "C" int lstm_test_heads_timeout(int withhold, unsigned int wait_limit_us, int device)
{
    return set_timeout_test(kTestHeads, "heads", withhold, wait_limit_us, device);
}
