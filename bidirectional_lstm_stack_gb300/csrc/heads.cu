// The dense heads of the segmentation model on the LSTM stack's output
// (speakrs 0.6.0 pages, segdense.rs: `Site::Linear0` a row-major 256-to-128
// projection `[k, n]` with bias and LeakyReLU, `Site::Linear1` 128-to-128 with
// bias and LeakyReLU, `Site::Linear2` 128-to-7 with bias and log-softmax;
// `DenseOxide`: those epilogues fused into the GEMMs), per row of y:
//     h1 = leaky(y W0 + b0),  h2 = leaky(h1 W1 + b1),
//     out = log_softmax(h2 W2 + b2)  (7 classes).
//
// Each layer is one launch of the tensor-core GEMM of projection.cu (3xTF32,
// persistent, 2-CTA clusters sharing each W tile by multicast) with its
// epilogue fused: bias and LeakyReLU on the accumulator before the TMA store
// of h1 / h2, or bias and log-softmax over the 7 class logits of a row,
// written directly.  h1 and h2 are [rows][128] scratch the object owns.  The
// weights are packed once at create: transposed to [n][k] (the K-major B
// operand) and split into TF32 hi/lo planes; the classifier's 7 output rows
// are padded to the 16-row MMA tile with zeros.
#include <stdlib.h>
#include <string.h>

#include <new>

#include "common.cuh"

using namespace lstm;

namespace {
constexpr int kIn = LSTM_STACK_OUTPUT;      // 256
constexpr int kMid = LSTM_HEADS_HIDDEN;     // 128
constexpr int kCls = LSTM_HEADS_CLASSES;    // 7
constexpr int kClsRows = 16;                // classifier MMA tile (N)
}  // namespace

struct lstm_heads {
    int device = 0;
    long max_rows = 0;
    float slope = 0.01f;
    float *weights = nullptr;  // one allocation: packed planes and biases
    float *w_hi[3] = {}, *w_lo[3] = {}, *bias[3] = {};
    float *h1 = nullptr, *h2 = nullptr;  // [max_rows][128]
    CUtensorMap map_whi[3], map_wlo[3];
    CUtensorMap load_h1, load_h2, store_h1, store_h2;
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
    cudaFree(h->h1);
    cudaFree(h->h2);
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

    // layer l: source W [K][N] row-major ([k, n]), packed [Npad][K]
    const float *src_w[3] = {w0, w1, w2};
    const float *src_b[3] = {b0, b1, b2};
    const int K[3] = {kIn, kMid, kMid};
    const int N[3] = {kMid, kMid, kCls};
    const int Npad[3] = {kMid, kMid, kClsRows};
    long off_hi[3], off_lo[3], off_b[3], total = 0;
    for (int l = 0; l < 3; ++l) {
        off_hi[l] = total;  total += static_cast<long>(Npad[l]) * K[l];
        off_lo[l] = total;  total += static_cast<long>(Npad[l]) * K[l];
        off_b[l] = total;   total += Npad[l];
        total = (total + 63) / 64 * 64;  // every plane 256-byte aligned
    }
    float *host = static_cast<float *>(calloc(total, sizeof(float)));
    if (!host) {
        lstm_heads_destroy(h);
        return fail(LSTM_E_ALLOC, "lstm_heads_create: host staging allocation failed");
    }
    for (int l = 0; l < 3; ++l) {
        for (int n = 0; n < N[l]; ++n) {
            for (int k = 0; k < K[l]; ++k) {
                const float v = src_w[l][static_cast<long>(k) * N[l] + n];
                const float hi = tf32_round(v);
                host[off_hi[l] + static_cast<long>(n) * K[l] + k] = hi;
                host[off_lo[l] + static_cast<long>(n) * K[l] + k] = tf32_round(v - hi);
            }
            host[off_b[l] + n] = src_b[l][n];
        }
    }
    cudaError_t e = device_alloc(reinterpret_cast<void **>(&h->weights), total * sizeof(float));
    if (e == cudaSuccess)
        e = cudaMemcpy(h->weights, host, total * sizeof(float), cudaMemcpyHostToDevice);
    free(host);
    if (e == cudaSuccess)
        e = device_alloc(reinterpret_cast<void **>(&h->h1), max_rows * kMid * sizeof(float));
    if (e == cudaSuccess)
        e = device_alloc(reinterpret_cast<void **>(&h->h2), max_rows * kMid * sizeof(float));
    if (e != cudaSuccess) {
        cudaGetLastError();
        lstm_heads_destroy(h);
        return fail(LSTM_E_ALLOC, "lstm_heads_create: device allocation: %s",
                    cudaGetErrorString(e));
    }
    const int box_rows[3] = {kHeadWBoxRows, kHeadWBoxRows, kClassifierWBoxRows};
    for (int l = 0; l < 3 && st == LSTM_OK; ++l) {
        h->w_hi[l] = h->weights + off_hi[l];
        h->w_lo[l] = h->weights + off_lo[l];
        h->bias[l] = h->weights + off_b[l];
        st = encode_matrix_map(&h->map_whi[l], h->w_hi[l], Npad[l], K[l], box_rows[l]);
        if (st == LSTM_OK)
            st = encode_matrix_map(&h->map_wlo[l], h->w_lo[l], Npad[l], K[l], box_rows[l]);
    }
    // the scratch maps cover max_rows: rows past a call's count are scratch
    // too, and the classifier writes only the call's rows
    if (st == LSTM_OK)
        st = encode_matrix_map(&h->load_h1, h->h1, max_rows, kMid, kProjectionBoxRows);
    if (st == LSTM_OK)
        st = encode_matrix_map(&h->load_h2, h->h2, max_rows, kMid, kProjectionBoxRows);
    if (st == LSTM_OK)
        st = encode_store_map(&h->store_h1, h->h1, max_rows, kMid);
    if (st == LSTM_OK)
        st = encode_store_map(&h->store_h2, h->h2, max_rows, kMid);
    if (st != LSTM_OK) {
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
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = launch_head_leaky(h->map_y, h->map_whi[0], h->map_wlo[0], h->store_h1, h->bias[0],
                                h->slope, rows, kIn, h->fault, s)))
        return st;
    if ((st = launch_head_leaky(h->load_h1, h->map_whi[1], h->map_wlo[1], h->store_h2,
                                h->bias[1], h->slope, rows, kMid, h->fault, s)))
        return st;
    return launch_head_classifier(h->load_h2, h->map_whi[2], h->map_wlo[2], h->bias[2], logp, rows,
                                  kMid, h->fault, s);
}
