/*
 * lstm_stack.h -- C ABI of liblstmstack.so, a GB300 (sm_103a) forward pass of
 * the four-layer bidirectional LSTM stack (hidden size 128, input width 60 for
 * the first layer and 256 after it, gate blocks i, f, g, o).
 *
 * The operation is the one the speakrs 0.6.0 pages define (docs.rs source of
 * src/inference/cuda/candidate/lstmproj.rs and lstm.rs):
 *  - module docs: per layer, a projection `x . W^T` for every step of each
 *    direction with the gate columns reordered so each hidden unit's four
 *    gates are adjacent, then one persistent recurrence per direction with
 *    the recurrent weights on chip; the reverse direction runs beside the
 *    forward one and the next layer waits for both;
 *  - `PackedLayer`: W `[2, padded_input, 512]`/`[2, 512, padded_input]`,
 *    R `[2, 512, 128]`, bias `[2, 512]` = Wb + Rb;
 *  - `Oxide::with_recurrence`, pack closure: source lengths W = 2*512*input,
 *    R = 2*512*128, B = 4*512;
 *  - `Oxide::enqueue`: input `rows * 60`, output `rows * 256`, rows =
 *    batch * steps; `check_len` / `to_u32`: exact-length and 32-bit checks;
 *  - `recur`: the reverse direction's h goes to output columns 128..255.
 * Cell equations (not printed on the pages; the standard LSTM):
 *   z = W x_t + Wb + R h_prev + Rb,  i = s(z_i), f = s(z_f), g = tanh(z_g),
 *   o = s(z_o),  c = f c + i g,  h = o tanh(c),  h and c start at zero.
 *
 * Conventions for every entry point below:
 *  - All floating-point data is IEEE fp32, row-major, densely packed.
 *  - "device" pointers are CUDA device (or managed) memory on the stack's
 *    device; "host" pointers are CPU memory (pinned memory makes the copies
 *    asynchronous).  Device pointers passed to a TMA-fed call must be 16-byte
 *    aligned (cudaMalloc and torch give 256-byte alignment).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Device work is enqueued on it asynchronously; nothing
 *    synchronises unless stated.
 *  - The return value is LSTM_OK (0) or one of the LSTM_E_* codes;
 *    lstm_stack_last_error() then returns a message for the calling thread.
 *    No C++ exception crosses this boundary.
 *  - Finite inputs give finite, bounded outputs (the activations' exponential
 *    saturates to 0 or infinity, so every gate stays in [0, 1]).  How NaN or
 *    infinite inputs surface is unspecified, as on the pages
 *    (`SPECIAL_VALUES`).
 */
#ifndef LSTM_STACK_H
#define LSTM_STACK_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LSTM_STACK_LAYERS 4
#define LSTM_STACK_HIDDEN 128
#define LSTM_STACK_FEATURES 60
#define LSTM_STACK_GATES 512         /* 4 * HIDDEN, one direction            */
#define LSTM_STACK_GATE_COLUMNS 1024 /* both directions' packed gate columns */
#define LSTM_STACK_OUTPUT 256        /* 2 * HIDDEN                           */

enum {
    LSTM_OK = 0,
    LSTM_E_INVALID = 1,  /* null pointer, non-positive or too-large size, bad direction, misaligned pointer */
    LSTM_E_LENGTH = 2,   /* a buffer length differs from what the sizes need (message: expected/actual) */
    LSTM_E_OVERFLOW = 3, /* a dimension does not fit the kernels' 32-bit indexing */
    LSTM_E_DEVICE = 4,   /* the device is not sm_103 / refuses a needed attribute */
    LSTM_E_CUDA = 5,     /* a CUDA runtime/driver call failed (message: its error string) */
    LSTM_E_ALLOC = 6,    /* host or device allocation failed */
    LSTM_E_FAULT = 7     /* a kernel's bounded wait ran out and it set its fault word */
};

/* How the input projection multiplies (lstmproj.rs `CudaMath` and
 * `projection_rule`).  LSTM_MATH_3XTF32 (default): three TF32 tensor-core
 * products per fp32 product (x_hi*w_hi + x_hi*w_lo + x_lo*w_hi), fp32-level
 * accuracy.  LSTM_MATH_TF32: one product of the operands rounded to TF32
 * (10 stored mantissa bits, to nearest, ties away), fp32 accumulation; a
 * third of the tensor work, with the TF32 rounding error the pages found too
 * large on some parts (`tf32_projection_accurate`).  The recurrence is fp32
 * in both. */
enum {
    LSTM_MATH_3XTF32 = 0,
    LSTM_MATH_TF32 = 1
};

/* ---------------------------------------------------------------------------
 * The stack (create / forward / destroy)
 * ------------------------------------------------------------------------- */

typedef struct lstm_stack lstm_stack; /* opaque; owned by the library */

/* Source weights, host fp32, read only during lstm_stack_create.  Layer l:
 *   w[l] : [2][512][in_l]  direction d's W, gate row blocks i,f,g,o
 *                          (row k*128 + u is gate k of unit u); in_0 = 60,
 *                          in_l = 256 for l >= 1
 *   r[l] : [2][512][128]   direction d's R, same row blocks
 *   b[l] : [2][1024]       direction d's Wb[512] followed by Rb[512]
 * Direction 0 is forward, 1 reverse. */
typedef struct {
    const float *w[LSTM_STACK_LAYERS];
    const float *r[LSTM_STACK_LAYERS];
    const float *b[LSTM_STACK_LAYERS];
} lstm_stack_weights;

/* Packs the weights (lstm_pack_layer) and copies them to `device`, allocates
 * the device scratch for up to max_batch windows of up to max_steps steps
 * (gate buffer [rows][1024], two ping-pong layer buffers [rows][256], two
 * staging slots [rows][60] + [rows][256] for the host-memory entry points),
 * creates the copy streams and the events.
 * On success *out owns all of it.  Errors: LSTM_E_INVALID (null, sizes <= 0),
 * LSTM_E_OVERFLOW (max_batch*max_steps*1024 beyond 2^31 rows*cols),
 * LSTM_E_DEVICE (device is not compute capability 10.3 or lacks cluster
 * launch), LSTM_E_CUDA, LSTM_E_ALLOC.  Nothing is leaked on failure. */
int lstm_stack_create(const lstm_stack_weights *weights, int max_batch,
                      int max_steps, int device, lstm_stack **out);

/* Gate order of the source row blocks of W, R, Wb and Rb.  The pages' source
 * layout (`Oxide::with_recurrence`: W [2][512][in], R [2][512][128],
 * B = per direction Wb ++ Rb) is ONNX-shaped; ONNX orders the blocks
 * i, o, f, c (c = the cell candidate g), PyTorch and this library's default
 * i, f, g, o. */
enum {
    LSTM_GATES_IFGO = 0,
    LSTM_GATES_IOFC = 1
};

/* lstm_stack_create for weights whose row blocks are in `gate_order`
 * (LSTM_GATES_IFGO or LSTM_GATES_IOFC); everything else as there.  Errors:
 * those of lstm_stack_create, and LSTM_E_INVALID for an unknown order. */
int lstm_stack_create_ordered(const lstm_stack_weights *weights, int gate_order,
                              int max_batch, int max_steps, int device,
                              lstm_stack **out);

/* y = stack(x) for `batch` independent windows of `steps` steps.
 *   x : device [batch][steps][60],  x_len = batch*steps*60 floats
 *   y : device [batch][steps][256], y_len = batch*steps*256 floats;
 *       y[b][t][0:128] forward h, y[b][t][128:256] reverse h
 * x and y must not overlap each other or the stack's scratch.  Enqueued on
 * `stream`; never allocates device memory and does not synchronise.  Each
 * layer runs its projection, then the forward and the reverse recurrence
 * together in one launch (the pages run the reverse one on a side stream
 * beside the forward one, `recur`); each projection may start while the
 * kernel before it ends and waits for it before touching its output
 * (programmatic dependent launch).  The work is replayed from a CUDA graph: the first
 * call with a given (x, y, batch, steps) records and instantiates the graph
 * (driver-side host resources; up to 8 argument sets are kept, least
 * recently used evicted), later calls launch it.  If `stream` is being
 * captured by the caller, the launches are enqueued directly into the
 * caller's capture instead.  Calls on one stack object must not overlap
 * (they share its scratch).  Errors: LSTM_E_INVALID (null, batch/steps <= 0
 * or above the create-time maxima, x not 16-byte aligned, device mismatch),
 * LSTM_E_LENGTH, LSTM_E_CUDA. */
int lstm_stack_forward(lstm_stack *s, const float *x, size_t x_len, float *y,
                       size_t y_len, int batch, int steps, void *stream);

/* The same forward pass from and to host memory, without waiting for it:
 * copies x (host, x_len floats) into one of the stack's two device staging
 * slots on an internal input-copy stream, runs the forward on `stream`, and
 * copies the result into y (host, y_len floats) on an internal output-copy
 * stream.  Consecutive calls use the two slots in turn, so one call's output
 * copy and the next call's input copy overlap the next forward; a call
 * reuses a slot only after that slot's previous output copy, and starts its
 * forward only after the previous call's forward (the stack's scratch is
 * shared).  x must stay unchanged until the call's input copy is done and y
 * is valid after lstm_stack_host_sync; both should be page-locked (pinned)
 * for the copies to be asynchronous.  As with lstm_stack_forward, calls on
 * one stack object must not overlap in time on the host.  Not for a stream
 * being captured
 * (LSTM_E_INVALID; capture lstm_stack_forward instead).  Errors: those of
 * lstm_stack_forward, LSTM_E_INVALID for a capturing stream. */
int lstm_stack_forward_host_async(lstm_stack *s, const float *x_host, size_t x_len,
                                  float *y_host, size_t y_len, int batch,
                                  int steps, void *stream);

/* Waits for every lstm_stack_forward_host_async call enqueued so far (their
 * output copies, hence their forwards).  Returns LSTM_E_FAULT if a kernel of
 * one of them reported a bounded wait that ran out (the results are not
 * valid; the fault word is cleared), else LSTM_OK or LSTM_E_CUDA. */
int lstm_stack_host_sync(lstm_stack *s);

/* lstm_stack_forward_host_async followed by lstm_stack_host_sync: y is ready
 * on return (LSTM_E_FAULT as there). */
int lstm_stack_forward_host(lstm_stack *s, const float *x_host, size_t x_len,
                            float *y_host, size_t y_len, int batch, int steps,
                            void *stream);

/* Opt-in per-phase timing (the pages' `LstmPhases` hooks): when enabled,
 * every forward records CUDA events around each layer's projection and
 * around its recurrence (both on the caller's stream).  lstm_stack_phase_times
 * then waits for the last forward and writes 12 milliseconds into ms[12]: for
 * layer l, ms[3l] projection, ms[3l+1] and ms[3l+2] the recurrence (both
 * directions run in one launch, so the two slots hold the same time).  The
 * events sit between kernels that otherwise overlap their set-up with the
 * previous kernel's tail, so a timed forward runs a little slower. */
int lstm_stack_enable_phase_timing(lstm_stack *s, int enable);
int lstm_stack_phase_times(lstm_stack *s, float *ms);

/* Turns graph replay in lstm_stack_forward(_host) on (default) or off
 * (direct launches every call); results are identical either way. */
int lstm_stack_set_graphs(lstm_stack *s, int enable);

/* Selects the projection's products for the following forward passes:
 * LSTM_MATH_3XTF32 (default) or LSTM_MATH_TF32.  Errors: LSTM_E_INVALID
 * (null stack, unknown mode). */
int lstm_stack_set_math(lstm_stack *s, int math);

/* Forward passes with batch <= max_batch compute each layer's input
 * projection inside its recurrence (lstm_recurrence_fused: no projection
 * kernel, no gate buffer round trip; the pages' SURVEY-ranked follow-on for
 * one window, the input projection of lstmproj.rs module docs folded into
 * `recur`); larger batches, and max_batch 0 (the default), run the
 * projection kernel and the recurrence, and so do batches whose clusters
 * (8 CTAs of 256 threads per window and direction) the device cannot run all
 * at once.  The fused products are fp32 FMAs, so results differ from the
 * default path in the last bits.  Errors: LSTM_E_INVALID (null,
 * max_batch < 0). */
int lstm_stack_set_fused_batches(lstm_stack *s, int max_batch);

/* Releases everything the stack owns (waits for its pending work first).
 * NULL is ignored. */
void lstm_stack_destroy(lstm_stack *s);

/* Message for the calling thread's last failed call ("" if none). */
const char *lstm_stack_last_error(void);

/* ---------------------------------------------------------------------------
 * The steps of the path, exposed one by one (used by the stack above; also
 * callable on their own for testing and measurement)
 * ------------------------------------------------------------------------- */

/* Step 1, host: gate-interleaving packer of one layer (lstmproj.rs module
 * docs and `PackedLayer`).  Host-only; needs no GPU.
 *   w : [2][512][in_width], r : [2][512][128], b : [2][1024] (source layout)
 *   wp_hi, wp_lo : [1024][kp]  both directions' W stacked; packed row
 *        n = d*512 + 4u + k holds source row k*128 + u of direction d,
 *        columns in_width..kp-1 zero; wp_hi is that value rounded to TF32
 *        (round to nearest, ties away) and wp_lo = value - wp_hi, also
 *        rounded to TF32, so wp_hi + wp_lo carries fp32-level precision
 *   rp : [2][512][128]  packed row 4u + k of direction d = source row k*128+u
 *   bias : [2][512]     bias[d][4u + k] = Wb[d][k*128+u] + Rb[d][k*128+u] (fp32)
 * kp must be >= in_width and a multiple of 32.  Errors: LSTM_E_INVALID. */
int lstm_pack_layer(const float *w, const float *r, const float *b,
                    int in_width, int kp, float *wp_hi, float *wp_lo,
                    float *rp, float *bias);

/* lstm_pack_layer for source blocks in `gate_order` (LSTM_GATES_*): packed
 * row d*512 + 4u + k (k = 0..3 for i, f, g, o) takes the source row of gate k
 * of unit u in that order (for LSTM_GATES_IOFC: i from block 0, f from 2,
 * g from 3, o from 1), and likewise for R and the bias.  Errors:
 * LSTM_E_INVALID (as lstm_pack_layer, or an unknown order). */
int lstm_pack_layer_ordered(const float *w, const float *r, const float *b,
                            int in_width, int kp, int gate_order, float *wp_hi,
                            float *wp_lo, float *rp, float *bias);

/* Step 2, device: the input projection of one layer for both directions,
 *   g[m][n] = sum_j x[m][j] * wp[n][j],  m < rows, n < 1024,
 * computed on the tensor cores in a 3xTF32 split (x_hi*w_hi + x_hi*w_lo +
 * x_lo*w_hi with fp32 accumulation), so the result carries fp32-level
 * accuracy.  No bias is added.
 *   x : device [rows][in_width], rows of in_width floats (in_width*4 bytes
 *       must be a multiple of 16: 60 and 256 are)
 *   wp_hi, wp_lo : device [1024][kp] from lstm_pack_layer (kp = in_width
 *       rounded up to a multiple of 32; 64 for 60)
 *   g : device [rows][1024]
 * Errors: LSTM_E_INVALID (null, rows <= 0, in_width not in (0, kp], kp not a
 * multiple of 32, misaligned pointers), LSTM_E_OVERFLOW, LSTM_E_DEVICE,
 * LSTM_E_CUDA. */
int lstm_projection(const float *x, int rows, int in_width,
                    const float *wp_hi, const float *wp_lo, int kp, float *g,
                    void *stream);

/* lstm_projection with a chosen product (see LSTM_MATH_*): with
 * LSTM_MATH_TF32 it computes g[m][n] = sum_j tf32(x[m][j]) * wp_hi[n][j]
 * (wp_hi is already W rounded to TF32) with fp32 accumulation, and wp_lo is
 * not read (it may be NULL).  Errors: those of lstm_projection, and
 * LSTM_E_INVALID for an unknown mode. */
int lstm_projection_math(const float *x, int rows, int in_width,
                         const float *wp_hi, const float *wp_lo, int kp, float *g,
                         int math, void *stream);

/* The direction argument of the recurrence entry points: 0 forward, 1
 * reverse, or both in one launch (the stack's choice: forward and reverse
 * clusters alternate in one grid). */
#define LSTM_BOTH_DIRECTIONS 2

/* Step 3, device: one direction's recurrence over one layer.
 *   g    : device [batch*steps][1024] projection from lstm_projection
 *          (row b*steps + t); this direction reads columns d*512 .. d*512+511
 *   rp   : device [512][128]  this direction's packed R (lstm_pack_layer)
 *   bias : device [512]       this direction's packed bias
 *   y    : device [batch][steps][256]; writes columns d*128 .. d*128+127 only
 *   direction : 0 forward (t = 0..steps-1), 1 reverse (t = steps-1..0), or
 *          LSTM_BOTH_DIRECTIONS: both in one launch, rp then [2][512][128]
 *          and bias [2][512] (both directions as lstm_pack_layer writes them)
 *          and all 256 columns of y written
 * h and c start at zero for every window.  One thread-block cluster holds R
 * in its blocks' registers, split by hidden unit, and exchanges h through
 * distributed shared memory each step; the variant (cluster shape and
 * windows per cluster) is chosen from the batch size.  g, rp and y must be
 * 16-byte aligned (h is stored four units at a time).  Errors:
 * LSTM_E_INVALID (null, sizes, direction, alignment), LSTM_E_OVERFLOW,
 * LSTM_E_DEVICE, LSTM_E_CUDA. */
int lstm_recurrence(const float *g, const float *rp, const float *bias,
                    float *y, int batch, int steps, int direction,
                    void *stream);

/* lstm_recurrence with an explicit kernel variant, for tests and tuning.
 * A cluster of cluster_size blocks splits the 128 hidden units; each 8-lane
 * group of a block holds one unit's weights for a K chunk and runs `chunks`
 * independent chunks of windows_per_chunk windows.  Windows per cluster =
 * (threads_per_block / 8) / (128 / cluster_size) * windows_per_chunk * chunks.
 * threads_per_block 0 selects the default (256; 512 for clusters of 2).
 * Variants (cluster, windows_per_chunk, chunks, threads): (16|8, 1|2|4|8, 1,
 * 0), (4, 1|2|4|8, 1, 0), (2, 1, 1, 0), (4, 1, 2|4|8, 0), (4, 2, 2|4|8, 0),
 * (4, 4, 2|4, 0), (4, 8, 2, 0), (8, 2, 4, 0), and the narrow
 * (8, 1|2|4|8, 1, 128), (16, 1|2, 1, 64); and the two-unit variants, where
 * each 8-lane group holds two units' weights for a K chunk, so windows per
 * cluster = windows_per_chunk * chunks: (8, 1, 1, 64), (8, 4|8, 1|2, 64)
 * and (4, 4, 1|2, 128), (4, 8, 1, 128).  Every one of these
 * variants computes the same sums in the same order, so all give bitwise
 * identical y (the pages' three recurrence kernels are likewise bitwise
 * identical, lstmproj.rs module docs).  The variant (4, 16, 1, 128) runs the
 * matrix-vector products on the tensor cores instead (tcgen05.mma kind::tf32
 * in three TF32 products, R resident in tensor memory, 16 windows per
 * cluster of 4 CTAs): other summation order, so it matches the others to
 * rounding rather than bitwise; slower than the FFMA variants at every batch
 * on GB300, so never chosen by lstm_recurrence.  Errors as lstm_recurrence,
 * plus LSTM_E_INVALID for an unknown variant. */
int lstm_recurrence_variant(const float *g, const float *rp, const float *bias,
                            float *y, int batch, int steps, int direction,
                            int cluster_size, int windows_per_chunk, int chunks,
                            int threads_per_block, void *stream);

/* Step 2+3 fused, device, for small batches: one layer's recurrence that
 * computes its own input projection.  Each cluster (8 CTAs of 256 threads)
 * runs one window; half of each CTA's threads hold the layer's input weights
 * for the CTA's units (W = wp_hi + wp_lo, the packed planes) and, running
 * ahead of the recurrence, turn every step's input row into partial sums
 * that the recurrence lanes add to theirs before the reduction, so
 * z = W x_t + R h + bias with no G buffer (lstmproj.rs module docs: the
 * projection of every step, then the recurrence).
 *   x     : device [batch][steps][in_width], in_width a multiple of 4, <= kp
 *           (the layer input: the stack input or the previous layer's y)
 *   wp_hi, wp_lo : device [1024][kp], kp 64 or 256 (lstm_pack_layer)
 *   rp, bias, y, batch, steps, direction : as lstm_recurrence
 * The products are fp32 FMAs (not 3xTF32).  All clusters must run at once:
 * batch (times 2 for LSTM_BOTH_DIRECTIONS) at most the clusters the device
 * holds (LSTM_E_INVALID otherwise).  Errors as lstm_recurrence. */
int lstm_recurrence_fused(const float *x, int in_width, const float *wp_hi,
                          const float *wp_lo, int kp, const float *rp,
                          const float *bias, float *y, int batch, int steps,
                          int direction, void *stream);

/* Measurement: the recurrence's per-step latency floor.  Launches exactly
 * what lstm_recurrence launches for this batch (same variant, grid, cluster
 * and block shape, projection prefetch, distributed-shared-memory h
 * exchange, y stores and bounded waits), with the step's arithmetic -- the
 * 512 x 128 matrix-vector product, the reduction across lanes and the cell
 * update (lstmproj.rs module docs: the work each step of the persistent
 * recurrence does) -- replaced by a trivial dependence of each new h on one
 * received h value and the projection value.  Its time per step is the
 * latency the exchange alone sets, the floor the real kernel is measured
 * against.  Arguments, layout and errors as lstm_recurrence; y receives
 * meaningless values. */
int lstm_recurrence_floor(const float *g, const float *rp, const float *bias,
                          float *y, int batch, int steps, int direction,
                          void *stream);

/* Measurement: the dense rate of the tensor cores in the mode the projection
 * and the dense heads use (tcgen05.mma kind::tf32, M = 128, N = 256, K = 8,
 * fp32 accumulation in tensor memory).  One block per SM of `device` issues
 * 2 * `iterations` back-to-back MMAs on operands resident in shared memory;
 * the run is timed with CUDA events after a warm-up launch and *tflops
 * receives the TF32 rate (2*M*N*K flops per MMA).  The projection's 3xTF32
 * mode (three products per fp32 product, the split the pages choose for
 * fp32-level accuracy on the TF32 tensor path, segdense.rs "3xTF32") is
 * bound by a third of it.  Synchronises; allocates no device memory.
 * Errors: LSTM_E_INVALID (null, iterations outside 1..10^7), LSTM_E_DEVICE,
 * LSTM_E_CUDA, LSTM_E_FAULT (the kernel's bounded wait ran out). */
int lstm_tf32_rate(int device, int iterations, double *tflops);

/* How many clusters of a recurrence variant (as above) `device` can run at
 * once (cudaOccupancyMaxActiveClusters).  Errors: LSTM_E_INVALID (null,
 * unknown variant), LSTM_E_DEVICE, LSTM_E_CUDA. */
int lstm_recurrence_max_clusters(int cluster_size, int windows_per_chunk,
                                 int chunks, int threads_per_block, int device,
                                 int *max_clusters);

/* One bidirectional layer (projection, then the forward and the reverse
 * recurrence, all on `stream`) that allocates no device memory.  The paper
 * has no counterpart: this entry point exists for callers that cannot call
 * cudaMalloc -- code running under CUDA graph capture, plug-ins whose host
 * framework owns all device memory, loops that cannot afford an
 * allocation's implicit synchronisation.
 *   x      : device [batch][steps][in_width]
 *   wp_hi, wp_lo : device [1024][kp], rp : device [2][512][128],
 *   bias   : device [2][512]   (lstm_pack_layer's outputs, uploaded by the caller)
 *   y      : device [batch][steps][256] (forward h in columns 0..127,
 *            reverse h in 128..255)
 * The gate buffer between the projection and the recurrences is a fixed
 * 16 MiB file-scope device array (4096 rows of 1024 floats) that every GPU
 * loading the library holds until exit: batch*steps above 4096 is rejected
 * with LSTM_E_INVALID.  The first call on a device resolves the array's
 * address and sets kernel attributes, so make it before any stream
 * capture.  All calls share the array: calls that overlap on the GPU race
 * and must be ordered by the caller; it keeps the last call's contents, and
 * nothing in it needs clearing (each call writes every row it reads).
 * Every buffer must be on the current device and 16-byte aligned.  Errors:
 * LSTM_E_INVALID, LSTM_E_DEVICE, LSTM_E_CUDA. */
int lstm_layer_forward_static(const float *x, int batch, int steps,
                              int in_width, const float *wp_hi,
                              const float *wp_lo, int kp, const float *rp,
                              const float *bias, float *y, void *stream);

/* Reads and clears the library's device fault word on the current device
 * (set by a kernel whose bounded wait ran out; 0 = none).  Synchronises the
 * device. */
int lstm_fault_status(unsigned int *fault);

/* ---------------------------------------------------------------------------
 * Dense heads of the segmentation model on the stack output (segdense.rs,
 * `Site::Linear0` / `Linear1` / `Linear2` and `DenseOxide`, which fuses the
 * bias, LeakyReLU and log-softmax epilogues into the GEMMs).  For each row
 * m of y [rows][256] (a stack output row):
 *   h1 = leaky(y[m] W0 + b0),  h2 = leaky(h1 W1 + b1),
 *   logp[m] = log_softmax(h2 W2 + b2)  (7 classes),
 * leaky(v) = v for v >= 0, negative_slope * v below (the pages name the
 * activation without a slope; PyTorch's default is 0.01).  Every layer runs
 * on the tensor cores in 3xTF32 with fp32 accumulation.
 * ------------------------------------------------------------------------- */

#define LSTM_HEADS_HIDDEN 128
#define LSTM_HEADS_CLASSES 7

typedef struct lstm_heads lstm_heads; /* opaque; owned by the library */

/* Packs the weights (host fp32, read during the call only; row-major [k, n]
 * as the pages store them):
 *   w0 : [256][128], b0 : [128],  w1 : [128][128], b1 : [128],
 *   w2 : [128][7],   b2 : [7]
 * into device memory on `device` (W0 and W1 as TF32 hi/lo planes); the
 * forward keeps h1 and h2 on chip, so no activation buffer is allocated.
 * Errors: LSTM_E_INVALID (null, max_rows <= 0), LSTM_E_DEVICE, LSTM_E_CUDA,
 * LSTM_E_ALLOC.  Nothing is leaked on failure. */
int lstm_heads_create(const float *w0, const float *b0, const float *w1,
                      const float *b1, const float *w2, const float *b2,
                      float negative_slope, int max_rows, int device,
                      lstm_heads **out);

/* logp (device [rows][7]) = the heads on y (device [rows][256], 16-byte
 * aligned; e.g. lstm_stack_forward's output with rows = batch*steps),
 * asynchronously on `stream`; allocates nothing.  Calls on one object must
 * not overlap (they share its intermediate buffers).  Errors: LSTM_E_INVALID
 * (null, rows outside 1..max_rows, misaligned, wrong device), LSTM_E_LENGTH
 * (y_len != rows*256 or logp_len != rows*7), LSTM_E_CUDA. */
int lstm_heads_forward(lstm_heads *h, const float *y, size_t y_len, float *logp,
                       size_t logp_len, int rows, void *stream);

void lstm_heads_destroy(lstm_heads *h);

/* ---------------------------------------------------------------------------
 * Failure-injection hooks, for tests of the error paths without a GPU fault.
 * The pages have no counterpart.  Process-wide; not for production use.
 * ------------------------------------------------------------------------- */

/* After `skip` more device allocations by the library, the next `count` fail
 * as if cudaMalloc had run out of memory (the calls then return
 * LSTM_E_ALLOC and free what they had allocated).  count 0 turns it off. */
int lstm_test_fail_allocations(int skip, int count);

/* After `skip` more kernel launches by the library, the next `count` fail
 * with LSTM_E_CUDA ("injected launch failure") instead of launching; the
 * stack stays usable.  count 0 turns it off. */
int lstm_test_fail_launches(int skip, int count);

/* On `device`: with withhold != 0, CTA 0 of every recurrence cluster stops
 * pushing its hidden state, so its peers' per-step waits run out; every
 * recurrence wait gives up after wait_limit_us microseconds (at most 2 s;
 * 0 = the default 2 s).  A wait that runs out sets the fault word
 * (lstm_fault_status; lstm_stack_forward_host returns LSTM_E_FAULT), stops
 * waiting and lets the kernel finish: the context stays usable.  (0, 0)
 * restores normal operation.  Errors: LSTM_E_INVALID, LSTM_E_DEVICE,
 * LSTM_E_CUDA. */
int lstm_test_recurrence_timeout(int withhold, unsigned int wait_limit_us, int device);

/* The same for the projection (lstm_projection, and every projection the
 * stack runs): with withhold != 0 the kernel's TMA producer loads nothing, so
 * the waits of the warps that consume its stages run out; every wait gives
 * up after wait_limit_us (at most 2 s; 0 = 2 s).  A wait that runs out sets
 * the fault word, every role of the kernel stops, drains what it issued,
 * frees its tensor memory and returns.  (0, 0) restores normal operation.
 * Errors as lstm_test_recurrence_timeout. */
int lstm_test_projection_timeout(int withhold, unsigned int wait_limit_us, int device);

/* The same for the dense heads (lstm_heads_forward). */
int lstm_test_heads_timeout(int withhold, unsigned int wait_limit_us, int device);

#ifdef __cplusplus
}
#endif

#endif /* LSTM_STACK_H */
