// Internal helpers shared by the library's translation units: error
// reporting across the C ABI, and thin inline-PTX wrappers for the sm_103a
// features the kernels use (mbarrier, TMA bulk tensor copies, tcgen05 /
// tensor memory, thread-block clusters and distributed shared memory).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lstm_stack.h"

namespace lstm {

constexpr int kHidden = LSTM_STACK_HIDDEN;          // 128
constexpr int kGates = LSTM_STACK_GATES;            // 512 per direction
constexpr int kGateColumns = LSTM_STACK_GATE_COLUMNS; // 1024, both directions
constexpr int kFeatures = LSTM_STACK_FEATURES;      // 60
constexpr int kOutput = LSTM_STACK_OUTPUT;          // 256

// Records a message for lstm_stack_last_error() and returns `code`.
int fail(int code, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
// Maps a CUDA error to LSTM_E_CUDA with its string; LSTM_OK on success.
int cuda_status(cudaError_t err, const char *what);

// Fault bits a kernel sets in the library's device fault word when one of
// its bounded waits runs out.
enum : unsigned {
    kFaultProducer = 1u << 0,
    kFaultConverter = 1u << 1,
    kFaultMma = 1u << 2,
    kFaultEpilogue = 1u << 3,
    kFaultDrain = 1u << 4,
    kFaultRecurrence = 1u << 5,
};

// The device fault word of the current device (a __device__ variable;
// resolved per device on first use).
unsigned *fault_word();

// ---- host helpers (api.cu) -------------------------------------------------
// Round-to-nearest (ties away from zero) to TF32: keep 10 mantissa bits.
float tf32_round(float x);
// Checks the device (cc 10.3, cluster launch) and sets the kernels'
// per-device attributes, once per device.
int prepare_device(int device);
// cudaMalloc, or an injected cudaErrorMemoryAllocation while the
// lstm_test_fail_allocations counter is positive.
cudaError_t device_alloc(void **p, size_t bytes);
// LSTM_E_CUDA (an injected launch failure) while the lstm_test_fail_launches
// counter is positive, else LSTM_OK; every kernel launch asks first.
int check_launch_injection(const char *what);
// Failure-test settings of one kernel on one device, passed to its launches
// as kernel parameters: every bounded wait gives up after wait_limit_ns, and
// with `withhold` the kernel starves its own waits (the recurrence: CTA 0 of
// every cluster pushes no h; the projection and the heads: the producer
// loads nothing).  Defaults: 2 s, no withholding.
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;
struct KernelTest {
    unsigned long long wait_limit_ns = kDefaultWaitLimitNs;
    int withhold = 0;
};
enum TestKernel { kTestRecurrence = 0, kTestProjection = 1, kTestHeads = 2, kTestKernels = 3 };
// The settings of `kernel` on the current device.
KernelTest kernel_test(int kernel);
// Sets them on the current device.
int set_kernel_test(int kernel, int withhold, unsigned long long wait_limit_ns);
// Whether any failure-test setting is in force on `device` (the stack then
// launches directly instead of replaying a graph captured without it).
bool kernel_test_active(int device);
// LSTM_E_INVALID unless p is 16-byte aligned.
int check_aligned(const void *p, const char *what);
// The device that owns device pointer p; LSTM_E_INVALID for host memory.
int pointer_device(const void *p, int *device);

// Makes `device` current for the scope and restores the previous one.
struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int device)
    {
        if (cudaGetDevice(&prev) != cudaSuccess)
            prev = -1;
        ok = (prev == device) || cudaSetDevice(device) == cudaSuccess;
    }
    ~DeviceGuard()
    {
        if (prev >= 0)
            cudaSetDevice(prev);
    }
};

// ---- projection (projection.cu) ------------------------------------------
// Rows per TMA box of the projection's operands: X rows, and the W gate rows
// of one tile (256, or 128 for the narrow tiles).
constexpr int kProjectionBoxRows = 128;
constexpr int kProjectionWBoxRows = 256;
constexpr int kProjectionNarrowWBoxRows = 128;
// Encodes the tensor map of a row-major fp32 matrix [rows][cols] read in
// boxes of 16 columns x box_rows rows with the 64-byte swizzle.
int encode_matrix_map(CUtensorMap *map, const float *base, long rows, int cols,
                      int box_rows);
// The tensor maps of one layer's packed W planes [1024][kp]: 256-row boxes
// for the 256-column tiles, 128-row boxes for the 128-column tiles used when
// few rows would leave most SMs idle.
struct ProjectionW {
    CUtensorMap hi, lo, hi_narrow, lo_narrow;
};
int encode_projection_w(ProjectionW *w, const float *wp_hi, const float *wp_lo, int kp);
// G[rows][1024] = X . Wp^T in 3xTF32 (math LSTM_MATH_3XTF32) or with single
// TF32 products (LSTM_MATH_TF32, the lo plane unused); x_map from
// encode_matrix_map (G's own store map is encoded per launch).
// grid_out (optional): the CTAs launched (the persistent grid).
int launch_projection(const CUtensorMap &x_map, const ProjectionW &w, float *g, int rows, int kp,
                      int math, unsigned *fault, cudaStream_t stream, int *grid_out = nullptr);
int projection_prepare(int device);
// Store map of a row-major fp32 matrix [rows][cols] written in 32 x 32
// slices with the 128-byte swizzle (the projection's G).
int encode_store_map(CUtensorMap *map, float *base, long rows, int cols);

// ---- dense heads of the segmentation model (heads.cu) ----------------------
// W rows of one k-block of the heads' weights (all 128 output columns).
constexpr int kHeadWBoxRows = 128;

// ---- recurrence (recurrence.cu) ------------------------------------------
// direction 0 (forward), 1 (reverse), or kBothDirections: one launch for
// both, rp [2][512][128] and bias [2][512], forward and reverse clusters
// alternating in the grid.
constexpr int kBothDirections = -1;
// co_resident_ctas >= 0: the kernel before it on the stream runs that many
// CTAs (the projection, one per SM); when both grids fit on the SMs side by
// side the recurrence is launched as its programmatic dependent, so its
// set-up (R into registers, barriers, the cluster barrier) overlaps that
// kernel, and it waits (griddepcontrol.wait) before it reads G.
int launch_recurrence(const float *g, const float *rp, const float *bias,
                      float *y, int batch, int steps, int direction,
                      unsigned *fault, cudaStream_t stream, int co_resident_ctas = -1);
int launch_recurrence_variant(const float *g, const float *rp, const float *bias,
                              float *y, int batch, int steps, int direction,
                              int cluster, int nw, int nch, int threads, unsigned *fault,
                              cudaStream_t stream);
// The default variant for `batch` in its FLOOR mode (the exchange alone:
// the step's arithmetic replaced by a trivial dependence on the received h).
int launch_recurrence_floor(const float *g, const float *rp, const float *bias, float *y,
                            int batch, int steps, int direction, unsigned *fault,
                            cudaStream_t stream);
// The recurrence with the projection fused in (small batches): x is the
// layer input [batch][steps][in_width] (in_width a multiple of 4, at most kp),
// wp_hi/wp_lo the layer's packed W planes [1024][kp] (kp 64 or 256); no G.
int launch_recurrence_fused(const float *x, int in_width, const float *wp_hi, const float *wp_lo,
                            int kp, const float *rp, const float *bias, float *y, int batch,
                            int steps, int direction, unsigned *fault, cudaStream_t stream);
// Clusters of the fused kernel (for kp) the device holds at once.
int recurrence_fused_max_clusters(int kp, int *out);
// Clusters of a variant the device can hold at once.
int recurrence_max_clusters(int cluster, int nw, int nch, int threads, int *out);
int recurrence_prepare(int device);

} // namespace lstm

// ---------------------------------------------------------------------------
// Device-side PTX wrappers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__
namespace lstm {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// fp32 rounded to TF32 (10 mantissa bits), nearest with ties away from zero.
__device__ __forceinline__ float tf32_rna(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier ----
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Waits for the phase with `parity` to complete, for at most `limit_ns`
// nanoseconds, or until *abort becomes non-zero.  Returns false (after
// setting `code` in *fault and *abort) when the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  volatile int *abort, unsigned *fault,
                                                  unsigned code, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t start = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*abort)
            return false;
        if (globaltimer() - start > limit_ns) {
            atomicOr(fault, code);
            *abort = 1;
            return false;
        }
    }
}

// ---- TMA ----
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
                 : "memory");
}
// Global -> this CTA's shared memory, `bytes` (a multiple of 16, both
// addresses 16-byte aligned), credited to `bar` as transaction bytes.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
// Shared memory -> global through the tensor map; the TMA engine writes only
// the part of the box inside the tensor.  Tracked by bulk groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// At most N of this thread's bulk groups still reading their shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// At most N of this thread's bulk groups not yet complete.
template <int N>
__device__ __forceinline__ void bulk_wait_group()
{
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- tcgen05 / tensor memory ----
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::tf32, one CTA.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}
// The same with A in tensor memory: A's rows are tensor-memory lanes, its K
// elements consecutive 32-bit columns starting at a_tmem.
__device__ __forceinline__ void mma_tf32_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}
// Arrives once on `bar` when every tcgen05 operation this thread issued
// before has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ uint32_t cluster_nid_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                 "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, "
                 "%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
                   "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]),
                   "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- clusters / distributed shared memory ----
// This CTA's shared memory -> the shared memory of a CTA of the cluster
// (`dst` and `remote_bar` cluster addresses from mapa), `bytes` a multiple of
// 16 with both addresses 16-byte aligned, credited to the peer's mbarrier as
// transaction bytes; read and written in the asynchronous proxy.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst, uint32_t src, uint32_t bytes,
                                                  uint32_t remote_bar)
{
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes"
                 " [%0], [%1], %2, [%3];" ::"r"(dst),
                 "r"(src), "r"(bytes), "r"(remote_bar)
                 : "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}
// One-sided push of four consecutive floats into a peer CTA's shared memory;
// on arrival the peer's mbarrier at `remote_bar` is credited with 16
// transaction bytes.
__device__ __forceinline__ void st_async_v4(uint32_t remote_addr, float a, float b, float c,
                                            float d, uint32_t remote_bar)
{
    // No "memory" clobber: the pushed buffer is read only after a wait on
    // its mbarrier, and that wait is the compiler barrier; leaving this store
    // unordered lets independent work be scheduled around it.
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     remote_addr),
                 "f"(a), "f"(b), "f"(c), "f"(d), "r"(remote_bar));
}
// try_wait with acquire semantics at cluster scope (pairs with the
// transaction credit of st.async from peer CTAs).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}
// Asynchronous 4-byte copy from global memory into this CTA's shared memory:
// `bytes` = 4, or 0 to zero the word without reading the source.  Copies of
// one thread complete in the order of their commit groups.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, uint32_t bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(bytes)
                 : "memory");
}
// The same for 16 bytes (both addresses 16-byte aligned; `bytes` 16 or 0),
// cached in L2 only.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}
// Waits until at most N of this thread's most recent commit groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}
// Programmatic dependent launch: wait until the grid this one depends on
// has completed and its memory is visible (returns at once when the kernel
// was launched without the dependency), and let the grid that depends on this
// one be scheduled before this one ends.
__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns from registers (thread = lane).
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                 "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
                 "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
                 "%32};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                 "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
                 "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
                 "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]),
                 "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// tcgen05 shared-memory matrix descriptor: K-major operand, 64-byte
// swizzle, 8-row groups 512 bytes apart.
__device__ __forceinline__ uint64_t sw64_desc(uint32_t addr)
{
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) |
           (static_cast<uint64_t>(1) << 16) |           // leading offset (unused, swizzled K-major)
           (static_cast<uint64_t>(512 >> 4) << 32) |    // stride offset: 8 rows x 64 B
           (static_cast<uint64_t>(1) << 46) |           // descriptor version (tcgen05)
           (static_cast<uint64_t>(4) << 61);            // 64-byte swizzle
}

// Instruction descriptor of kind::tf32, M = m, N = n: D fp32, A and B TF32,
// both K-major.
__host__ __device__ constexpr uint32_t tf32_idesc(int m, int n)
{
    return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

// Splits four fp32 values into TF32 hi parts and TF32 remainders.
__device__ __forceinline__ void split4(float4 v, float4 &hi, float4 &lo)
{
    hi.x = tf32_rna(v.x); lo.x = tf32_rna(v.x - hi.x);
    hi.y = tf32_rna(v.y); lo.y = tf32_rna(v.y - hi.y);
    hi.z = tf32_rna(v.z); lo.z = tf32_rna(v.z - hi.z);
    hi.w = tf32_rna(v.w); lo.w = tf32_rna(v.w - hi.w);
}

// Waits without regard to any abort flag, up to limit_ns (used to drain
// in-flight work before shared or tensor memory goes away).
__device__ __forceinline__ void mbar_wait_drain(uint64_t *bar, uint32_t parity, unsigned *fault,
                                                uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return;
    const uint64_t start = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - start > limit_ns) {
            atomicOr(fault, kFaultDrain);
            return;
        }
    }
}

} // namespace ptx
} // namespace lstm
#endif
