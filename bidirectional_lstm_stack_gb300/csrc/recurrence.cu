// One direction's recurrence over one LSTM layer (the persistent kernel the
// speakrs 0.6.0 pages launch per direction, lstmproj.rs module docs and
// `recur` / `launch`):
//     z_t = G[b, t, d*512 : d*512+512] + bias_d + Rp_d . h_prev
//     i = s(z[4u]), f = s(z[4u+1]), g = tanh(z[4u+2]), o = s(z[4u+3])
//     c = f*c + i*g,   h = o*tanh(c),   y[b, t, d*128 + u] = h
// for t = 0..T-1 (forward) or T-1..0 (reverse), h and c starting at zero.
//
// Design (sm_103a): one thread-block cluster of C CTAs per tile of windows.
// CTA `rank` owns hidden units [rank*128/C, (rank+1)*128/C); its slice of the
// recurrent matrix (the four gate rows of each of its units, 128 columns)
// lives in registers for the whole kernel: thread (slot, kc) holds the 4 x 16
// weights of one unit for K chunk kc (16 columns).  Each step:
//   1. every thread multiplies its weights with h_prev[kc*16 .. +16] of each
//      of its windows from shared memory (paired FMAs, __ffma2_rn); a thread
//      runs NCH independent chunks of NW windows, each phase below over all
//      chunks, so their latencies overlap (or, for two chunks of 4 or more
//      windows, chunk by chunk with a barrier pair per chunk, so one chunk's
//      exchange overlaps the other's arithmetic);
//   2. the 8 lanes sharing a unit reduce their partial sums by a fixed
//      butterfly (lane bits 2, 1, 0): a reduce-scatter that leaves each lane
//      its share of the unit's gate pre-activations;
//   3. add the prefetched projection value and the bias, apply the bounded
//      activations, gather the four gates of a window (shuffles), update c
//      and h (c stays in registers);
//   4. gather the h of the warp's four consecutive units, push them into the
//      next-step h buffer of every CTA of the cluster with one 16-byte
//      st.async each (distributed shared memory), which credits the
//      receiving CTA's mbarrier for that buffer with the bytes written, then
//      write them to y (one float4); padding windows past the batch send
//      nothing;
//   5. before reading a buffer, wait on its mbarrier: the phase completes when
//      all 128 x (tile) values of the step have landed.
// Two h buffers alternate by step parity.  The exchange is one-sided: no
// cluster-wide barrier per step, no global flag words, and no release fence
// (which would also wait for the in-flight projection prefetch loads).  Data
// dependence makes the double buffer safe: a CTA can only push step s+1's h
// once it holds every unit's h_s, i.e. once every warp of every CTA has
// finished reading the buffer it is about to overwrite.  Each wait is bounded
// in time; when one runs out the kernel records a fault bit and every thread
// that sees it leaves its step loop for the final cluster barrier (no stuck
// barrier is re-armed or credited again), so the kernel ends, with invalid
// results, instead of hanging.
// The arithmetic per (window, unit, gate) is the same for every cluster size
// and tile width (same K chunks, same pairing, same reduction tree), so all
// variants give bitwise-identical results.
//
// Kernels in this file: recurrence_kernel (one hidden unit per 8-lane group,
// the design above); recurrence_u2_kernel and recurrence_u2w_kernel (two
// units per 8-lane group: half the shared-memory loads of h per multiply-add;
// one, or 2, 4 or 8 windows per lane), bitwise identical to it;
// recurrence_fused_kernel (the input projection computed beside the
// recurrence, small batches, opt-in); recurrence_tc_kernel (the products on
// the tensor cores, slower at this shape, never chosen).  choose_variant
// picks a variant per batch from measured step times.
#include <algorithm>
#include <mutex>
#include <type_traits>
#include <utility>

#include "common.cuh"

namespace lstm {
namespace {

// Threads per CTA: 256 (8 warps); clusters of 2 use 512 so that a CTA's
// half of R (64 units) still fits in registers at 64 per thread.
template <int C>
constexpr int threads_for()
{
    return C == 2 ? 512 : 256;
}
constexpr int KC = 8;                 // K chunks = lanes per reduction group
constexpr int KLEN = 16;              // columns per chunk
constexpr int CHUNK_STRIDE = 20;      // padded chunk stride (conflict-free LDS.128)
constexpr int HROW = KC * CHUNK_STRIDE;  // floats per window in the h buffer
constexpr int PF = 4;                 // projection prefetch depth (steps)


// Activations through base-2 exponentials of pre-scaled arguments: the
// recurrent weights, the bias and the projection value of gate q are
// multiplied by k_q = -log2(e) (-2 log2(e) for the cell candidate) as they
// are loaded, so a step produces w = k_q z directly and
//   s(z) = 1 / (1 + 2^w),   tanh(z) = 2 s(2z) - 1 = 2 / (1 + 2^w) - 1.
// 2^w overflows to +inf for large w and 1/inf is 0, so every gate is in
// [0, 1] (the candidate in [-1, 1]) for every finite z, without a clamp.
constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float inv_one_plus_ex2(float w)
{
    return __fdividef(1.0f, 1.0f + ex2_approx(w));
}

// The cell update c' = f c + i g, with one fixed rounding order (the product
// i g rounded, then one fused multiply-add), so every kernel computes the
// same bits whatever the compiler would contract.
__device__ __forceinline__ float cell_update(float i, float f, float g, float c)
{
    return fmaf(f, c, __fmul_rn(i, g));
}

// One butterfly level: lanes that differ in `mask` exchange half of their
// N values; each keeps the sums for the half its mask bit selects.
// PERM: the lane whose mask bit is set holds its values in an order with the
// two halves swapped (the lane-dependent order of the partial sums set up
// at kernel start), so every lane keeps its lower half and sends its upper
// half, without selects.  Otherwise the values are in logical order and
// each lane selects.  Both add the same two values.
template <int N, bool PERM>
__device__ __forceinline__ void reduce_level(const float (&in)[N], float (&out)[N / 2], int mask,
                                             bool upper)
{
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        if constexpr (PERM) {
            out[i] = in[i] + __shfl_xor_sync(0xffffffffu, in[i + N / 2], mask);
        } else {
            const float keep = upper ? in[i + N / 2] : in[i];
            const float send = upper ? in[i] : in[i + N / 2];
            out[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
        }
    }
}

// f(integral_constant<0>) && f(integral_constant<1>) && ... for N terms,
// left to right, stopping at the first false: the compile-time index lets
// the body pick register arrays by position.
template <typename F, int... I>
__device__ __forceinline__ bool unrolled_all_impl(F &f, std::integer_sequence<int, I...>)
{
    return (f(std::integral_constant<int, I>{}) && ...);
}
template <int N, typename F>
__device__ __forceinline__ bool unrolled_all(F &&f)
{
    return unrolled_all_impl(f, std::make_integer_sequence<int, N>{});
}

// FLOOR: the same kernel with the matrix-vector product, the reduction and
// the cell update replaced by a trivial dependence of each new h on the
// received h and on the projection value (same launch shape, projection
// prefetch, h gathers, st.async pushes, y stores and bounded waits): its time
// per step is the latency floor the exchange sets, which the bench reports
// beside the real kernel's.  Its outputs are meaningless.
template <int C, int NW, int NCH = 1, int THREADS = threads_for<C>(), bool FLOOR = false>
__global__ void __launch_bounds__(THREADS, 1)
recurrence_kernel(const float *__restrict__ g, const float *__restrict__ rp_in,
                  const float *__restrict__ bias_in, float *__restrict__ y, int batch, int steps,
                  int dir_in, unsigned *fault, unsigned long long wait_limit_ns, int withhold)
{
    constexpr int U = kHidden / C;       // units per CTA
    constexpr int SLOTS = THREADS / 8;   // 8-lane groups per CTA
    constexpr int SPU = SLOTS / U;       // slots per unit
    constexpr int LW = NW * NCH;         // windows per slot: NCH chunks of NW
    constexpr int TW = SPU * LW;         // windows per tile (per cluster)
    constexpr int V = 4 * NW;            // partial sums per thread and chunk
    constexpr int HV = V >= 8 ? V / 8 : 1;  // values a lane holds after the reduction
    constexpr int REPL = V >= 8 ? 4 / HV : 8;  // lanes holding one window's cell
    // Steps per unrolled group (the buffer parity and the prefetch slot are
    // compile-time within it), and the depth of the register ring of
    // projection values where that ring is used (see SRING below).  Measured
    // per step (GB300, T = 589) with the register ring, against 4 steps
    // ahead: 8 is 2 % faster at one window per chunk (2 steps: 8 % slower),
    // 1-2 % with 4 windows in one chunk, 4.5 % with two chunks of 2; it was
    // 1 % slower with one chunk of 2 and 4 % slower chunk-major.  Four or more
    // chunks: 2 (registers).  The shared-memory ring variants keep these
    // group lengths (one window: 8 measured better than 4 there too).
    constexpr bool DEEP = NW == 1 || (NW == 4 && NCH == 1) || (NW == 2 && NCH == 2);
    constexpr int PFD = NCH >= 4 ? 2 : (DEEP ? 2 * PF : PF);
    // Select-free butterfly (lane-dependent order of the partial sums) for
    // one window per chunk and for eight: measured faster there (GB300,
    // T = 589: 0.45 -> 0.40 us per step at one window, 2.61 -> 2.54 at 256
    // windows); with 2 or 4 windows per chunk it raised register use and
    // step time, so those keep the selects.
    constexpr bool PERM = NW == 1 || NW == 8;
    static_assert(U * SPU == SLOTS && C * U == kHidden && U % 4 == 0, "cluster shape");
    static_assert(PFD % 2 == 0, "the step parity is taken from the unrolled step index");
    // Chunk-major steps (CM): each chunk has its own pair of barriers and runs
    // all its phases before the next chunk starts, so a chunk's h exchange is
    // in flight while the next chunks compute.  Otherwise one barrier pair
    // covers the tile and each phase runs over all chunks, so their latencies
    // overlap.  Measured (GB300, T = 589): chunk-major is 9 % faster per step
    // with two chunks of 4 or 8 windows, and slower with smaller or more
    // chunks (the phases of one small chunk leave too little independent
    // work; four chunks of 4 windows: 4 % slower).
    constexpr bool CM = NCH == 2 && NW >= 4;
    // At most two chunks, where at least 4 steps fit: the projection values
    // travel through a ring in shared memory, filled by each lane's own
    // asynchronous copies GD steps ahead (no registers held for the values
    // in flight; measured per step against the register ring 8 steps ahead:
    // 4 % faster at one window, 1.5 % at 32 windows; with two windows per
    // chunk 5.5 % faster than 4 or 8 steps ahead); otherwise through a
    // register ring PFD steps ahead.  GD_FIT: ring slots that fit beside the
    // h buffers in 44 KiB of static shared memory (the static limit is
    // 48 KiB).
    constexpr int GD_FIT = (45056 - 2 * TW * HROW * 4) / (NCH * HV * THREADS * 4);
    constexpr int GD = GD_FIT >= 64   ? 64
                       : GD_FIT >= 32 ? 32
                       : GD_FIT >= 16 ? 16
                       : GD_FIT >= 8  ? 8
                                      : 4;
    constexpr bool SRING = NCH <= 2 && GD_FIT >= 4;
    constexpr int NBAR = CM ? NCH : 1;

    __shared__ __align__(16) float hbuf[2][TW][HROW];
    __shared__ __align__(8) uint64_t hbar[2][NBAR];
    __shared__ int abort_flag;
    __shared__ __align__(16) float gring[SRING ? GD : 1][SRING ? NCH * HV : 1][SRING ? THREADS : 1];

    const int tid = threadIdx.x;
    const int kc = tid & 7;
    const int slot = tid >> 3;
    // units vary fastest over slots, so the four 8-lane groups of a warp hold
    // four consecutive units of the same windows
    const int ul = slot % U;
    const int wg = slot / U;
    const uint32_t rank = ptx::cluster_ctarank();
    // one direction (dir_in 0 or 1), or both in one grid (dir_in < 0):
    // forward and reverse clusters alternate, each pair on one tile
    const int cid = static_cast<int>(ptx::cluster_id_x());
    const int direction = dir_in >= 0 ? dir_in : (cid & 1);
    const int tile = dir_in >= 0 ? cid : (cid >> 1);
    const float *__restrict__ rp = rp_in + (dir_in >= 0 ? 0 : direction * kGates * kHidden);
    const float *__restrict__ bias = bias_in + (dir_in >= 0 ? 0 : direction * kGates);
    const int u = static_cast<int>(rank) * U + ul;  // this thread's hidden unit
    const int wbase = wg * LW;                      // this slot's first window in the tile
    const int u0 = u & ~3;                          // first of the warp's four units
    // Padding windows (past the batch) are computed, but their h is neither
    // sent nor stored.  Bytes of one step's h per barrier: the tile's windows
    // inside the batch (chunk ch of every window group when chunk-major).
    uint32_t bar_bytes[NBAR];
    if constexpr (CM) {
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
            int n = 0;
            for (int grp = 0; grp < SPU; ++grp)
                n += max(0, min(NW, batch - (tile * TW + grp * LW + ch * NW)));
            bar_bytes[ch] = static_cast<uint32_t>(kHidden * n * 4);
        }
    } else {
        bar_bytes[0] = static_cast<uint32_t>(kHidden * min(TW, batch - tile * TW) * 4);
    }

    // The partial sums of a chunk have logical index w*4 + q (window w of
    // the chunk, gate q).  Lane kc keeps them in the order j -> j ^ xperm:
    // each butterfly level below then keeps the lower half of a lane's
    // array, which for a lane with that level's mask bit set is the upper
    // half of the logical values.  The order only permutes which gate row
    // and which window a slot computes; the sums and their order are the
    // same, so results do not depend on it.
    constexpr int X2 = V >= 8 ? V / 2 : 2, X1 = V >= 8 ? V / 4 : 1, X0 = V >= 8 ? V / 8 : 0;
    auto xperm_of = [](int k) {
        return PERM ? ((k & 4) ? X2 : 0) | ((k & 2) ? X1 : 0) | ((k & 1) ? X0 : 0) : 0;
    };
    // gate slot q holds gate q ^ xq; window slot w holds window w ^ (xperm >> 2)
    // of the chunk, which the senders realise by storing window w's values
    // of K chunk k at row w ^ (xperm_of(k) >> 2) of the chunk's rows, so
    // that slot w is read from row w
    const int xq = xperm_of(kc) & 3;

    // weights: 4 gate rows of unit u (slot q: gate q ^ xq), columns
    // kc*16 .. kc*16+15, as pairs, each row scaled by its gate's k_q (see the
    // activations above)
    float2 r2[4][KLEN / 2];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int gq_row = q ^ xq;
        const float kq = gq_row == 2 ? -2.0f * kLog2e : -kLog2e;
        const float2 *src =
            reinterpret_cast<const float2 *>(rp + (4 * u + gq_row) * kHidden + kc * KLEN);
#pragma unroll
        for (int i = 0; i < KLEN / 2; ++i)
            r2[q][i] = make_float2(src[i].x * kq, src[i].y * kq);
    }

    // The values this lane holds after each chunk's reduction: index
    // idx = w*4 + gate within the chunk (the same for every chunk).
    // Activations are branch-free across the lanes (which hold different
    // gates): act = m / (1 + 2^w) + a with (m, a) = (2, -1) for the cell
    // candidate and (1, 0) for the gates; w = k_q z = k_q (G + bias) +
    // (k_q R) h.
    float act_m[HV], act_a[HV], bias_v[HV], gk[HV];
    int wv[HV];
    const float *gcol[HV];
#pragma unroll
    for (int v = 0; v < HV; ++v) {
        const int idx = V >= 8 ? kc * HV + v : (kc >> 1);
        const int q = idx & 3;
        wv[v] = idx >> 2;
        gk[v] = q == 2 ? -2.0f * kLog2e : -kLog2e;
        bias_v[v] = bias[4 * u + q] * gk[v];
        act_m[v] = q == 2 ? 2.0f : 1.0f;
        act_a[v] = q == 2 ? -1.0f : 0.0f;
        gcol[v] = g + direction * kGates + 4 * u + q;
    }
    // the window (within a chunk) whose cell this lane updates; after the
    // gather below, the 4*REPL lanes of the warp that hold it share the sends
    // to the C CTAs
    const int wl = V >= 8 ? (kc * HV) / 4 : 0;
    const int sender = (tid & 31) / 8 * REPL + kc % REPL;  // 0 .. 4*REPL-1

    // h_{-1} = 0 in buffer 0; buffer 1 is zeroed too, so padding windows
    // (never sent) only ever see zeros
    for (int i = tid; i < 2 * TW * HROW; i += THREADS)
        (&hbuf[0][0][0])[i] = 0.0f;
    if (tid == 0) {
        for (int b = 0; b < NBAR; ++b) {
            ptx::mbar_init(&hbar[0][b], 1);
            ptx::mbar_init(&hbar[1][b], 1);
        }
        abort_flag = 0;
        ptx::fence_mbar_init();
        // arm buffer 1 for h_0 and buffer 0 for h_1.  A chunk with no window
        // inside the batch (chunk-major only) has no barrier traffic at all:
        // armed with zero bytes its phases would complete on every re-arm and
        // could run two phases ahead of a warp still waiting on the first.
        for (int b = 0; b < NBAR; ++b) {
            if (bar_bytes[b] == 0)
                continue;
            if (steps > 1)
                ptx::mbar_arrive_expect_tx(&hbar[1][b], bar_bytes[b]);
            if (steps > 2)
                ptx::mbar_arrive_expect_tx(&hbar[0][b], bar_bytes[b]);
        }
    }
    // every CTA of the cluster is running, zeroed and armed before anyone sends
    ptx::cluster_arrive_release();
    ptx::cluster_wait_acquire();

    const uint32_t hbase = ptx::smem_u32(&hbuf[0][0][0]);
    const uint32_t bar_base = ptx::smem_u32(&hbar[0][0]);
    const int tile_w0 = tile * TW;
    // chunk 0's projection column and output row; chunk ch is ch*NW windows on
    const long row_stride = static_cast<long>(NW) * steps;  // rows between chunks
    const float *gch0[HV];
#pragma unroll
    for (int v = 0; v < HV; ++v)
        gch0[v] = gcol[v] + static_cast<long>(tile_w0 + wbase + wv[v]) * steps * kGateColumns;
    float *ych0 = y + static_cast<long>(tile_w0 + wbase + wl) * steps * kOutput +
                  direction * kHidden + u0;
    const int bch0 = tile_w0 + wbase;  // window of chunk 0, w = 0
    // the four units u0..u0+3 lie in K chunk u0 / 16; their row within the
    // chunk's windows follows the readers' window order (see xperm_of)
    const uint32_t send_off0 = static_cast<uint32_t>(
        ((wbase + (wl ^ (xperm_of(u0 / KLEN) >> 2))) * HROW + (u0 / KLEN) * CHUNK_STRIDE +
         (u0 % KLEN)) *
        4);
    // the peers this lane sends to, and their h buffers and mbarriers for
    // both parities, as cluster addresses (a peer's shared memory is one
    // contiguous window, so offsets within it carry over)
    constexpr int NPEER = (C + 4 * REPL - 1) / (4 * REPL);
    uint32_t rdst[NPEER][2], rbar[NPEER][2];
#pragma unroll
    for (int r = 0; r < NPEER; ++r) {
        const int peer = min(sender + r * 4 * REPL, C - 1);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            rdst[r][q] = ptx::map_to_rank(
                hbase + static_cast<uint32_t>(q * TW * HROW * 4) + send_off0, peer);
            rbar[r][q] = ptx::map_to_rank(bar_base + static_cast<uint32_t>(q * NBAR * 8), peer);
        }
    }

    float gq[PFD][NCH][HV];
    // projection values of step s into dst; `check`: s may lie past the end
    auto gload = [&](int s, float (&dst)[NCH][HV], bool check) {
        const long t = direction ? steps - 1 - s : s;
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
#pragma unroll
            for (int v = 0; v < HV; ++v) {
                const bool ok = bch0 + ch * NW + wv[v] < batch && (!check || s < steps);
                dst[ch][v] = ok ? __ldg(gch0[v] + (ch * row_stride + t) * kGateColumns) : 0.0f;
            }
        }
    };
    // projection values of step s (one per chunk) into ring slot s % GD
    auto gissue = [&](int s) {
        const long t = direction ? steps - 1 - s : s;
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
#pragma unroll
            for (int v = 0; v < HV; ++v) {
                const bool ok = bch0 + ch * NW + wv[v] < batch && s < steps;
                const float *src = ok ? gch0[v] + (ch * row_stride + t) * kGateColumns : g;
                ptx::cp_async_4(ptx::smem_u32(&gring[s & (GD - 1)][ch * HV + v][tid]), src,
                                ok ? 4u : 0u);
            }
        }
        ptx::cp_async_commit();
    };
    // The next kernel (the next layer's projection, launched as a
    // programmatic dependent) may be scheduled from here on; it waits for
    // this one to end before it touches G or this layer's output.
    ptx::griddep_launch_dependents();
    // launched as a programmatic dependent of the kernel that writes its
    // input: wait for that kernel's end before the first read of it
    ptx::griddep_wait();
    if constexpr (SRING) {
        for (int s = 0; s < GD; ++s)
            gissue(s);
    } else {
#pragma unroll
        for (int p = 0; p < PFD; ++p)
            gload(p, gq[p], true);
    }

    float c[NCH];
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch)
        c[ch] = 0.0f;

    // The phases of a step for one chunk of NW windows, as the chunk-major
    // step runs them.  The phase-major step spells the same phases out inline
    // over all chunks: routed through these functions it measured 2 % slower
    // per step at one window per chunk.
    // 0. wait until the barrier's phase completes, false if the wait ran out
    //    or another warp's did: this thread then neither re-arms nor pushes
    //    again, so no stuck barrier is armed or credited after the fault.
    auto wait_phase = [&](uint64_t *bar, uint32_t phase) -> bool {
        volatile int *abort_v = &abort_flag;
        if (ptx::mbar_try_wait_cluster(bar, phase))
            return true;
        if (*abort_v)
            return false;
        const uint64_t start = ptx::globaltimer();
        while (!ptx::mbar_try_wait_cluster(bar, phase)) {
            if (*abort_v)
                return false;
            if (ptx::globaltimer() - start > wait_limit_ns) {
                atomicOr(fault, kFaultRecurrence);
                *abort_v = 1;
                return false;
            }
        }
        return true;
    };
    // 1. partial dot products of chunk ch over this lane's K chunk
    auto dots = [&](int par, int ch, float (&part)[V]) {
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float4 *hp = reinterpret_cast<const float4 *>(
                &hbuf[par][wbase + ch * NW + w][kc * CHUNK_STRIDE]);
            const float4 h0 = hp[0], h1 = hp[1], h2 = hp[2], h3 = hp[3];
            const float2 hh[8] = {{h0.x, h0.y}, {h0.z, h0.w}, {h1.x, h1.y}, {h1.z, h1.w},
                                  {h2.x, h2.y}, {h2.z, h2.w}, {h3.x, h3.y}, {h3.z, h3.w}};
            // the four gate rows' chains advance together (independent
            // FMAs back to back); each chain's order over i is fixed
            float2 acc[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                acc[q] = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    acc[q] = __ffma2_rn(r2[q][i], hh[i], acc[q]);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                part[w * 4 + q] = acc[q].x + acc[q].y;
        }
    };
    // 2. fixed butterfly over the 8 K-chunk lanes
    auto reduce = [&](const float (&part)[V], float (&held)[HV]) {
        if constexpr (V >= 8) {
            float a[V / 2], b2[V / 4];
            reduce_level<V, PERM>(part, a, 4, (kc & 4) != 0);
            reduce_level<V / 2, PERM>(a, b2, 2, (kc & 2) != 0);
            reduce_level<V / 4, PERM>(b2, held, 1, (kc & 1) != 0);
        } else {
            float a[2], b2[1];
            reduce_level<4, PERM>(part, a, 4, (kc & 4) != 0);
            reduce_level<2, PERM>(a, b2, 2, (kc & 2) != 0);
            held[0] = b2[0] + __shfl_xor_sync(0xffffffffu, b2[0], 1);
        }
    };
    // 3. activations, gate gather, cell update; returns h of window wl
    auto cell = [&](int ch, const float (&held)[HV], const float (&gv)[HV]) -> float {
        float act[HV];
#pragma unroll
        for (int v = 0; v < HV; ++v) {
            const float w = held[v] + fmaf(gv[v], gk[v], bias_v[v]);
            act[v] = fmaf(act_m[v], inv_one_plus_ex2(w), act_a[v]);
        }
        float gate[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int src = V >= 8 ? (4 * wl + q) / HV : 2 * q;
            gate[q] = __shfl_sync(0xffffffffu, act[q % HV], src, 8);
        }
        c[ch] = cell_update(gate[0], gate[1], gate[2], c[ch]);
        // h = o tanh(c) = o (2 r - 1) with r = 1 / (1 + 2^(-2 log2(e) c)):
        // one fused multiply-add after r
        const float r = inv_one_plus_ex2(c[ch] * (-2.0f * kLog2e));
        return fmaf(2.0f * gate[3], r, -gate[3]);
    };
    // 4. gather the warp's four units of window wl, push them (16 bytes)
    //    into every CTA's next h buffer (unless s is the last step) and store
    //    them to y
    auto emit = [&](int par, int ch, float h, bool push, int t) {
        float h4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            h4[j] = __shfl_sync(0xffffffffu, h, 8 * j + kc);
        if (bch0 + ch * NW + wl < batch) {
            if (push) {
                const uint32_t off = static_cast<uint32_t>(ch * NW * HROW * 4);
                const uint32_t bar_off = static_cast<uint32_t>(CM ? ch * 8 : 0);
#pragma unroll
                for (int r = 0; r < NPEER; ++r) {
                    if (sender + r * 4 * REPL < C)
                        ptx::st_async_v4(rdst[r][par ^ 1] + off, h4[0], h4[1], h4[2], h4[3],
                                         rbar[r][par ^ 1] + bar_off);
                }
            }
            if (sender == 0)
                *reinterpret_cast<float4 *>(ych0 + (ch * row_stride + t) * kOutput) =
                    make_float4(h4[0], h4[1], h4[2], h4[3]);
        }
    };

    // FLOOR: the new h of window wl depends on one received h value and on
    // the projection value, nothing else
    auto floor_h = [&](int par, int ch, const float (&gv)[HV]) -> float {
        const float hv = hbuf[par][wbase + ch * NW + wl][kc * CHUNK_STRIDE];
        return fmaf(hv, 0.5f, gv[0] * 0.001f);
    };

    // One step s (= s0 + P, P the position in the unrolled group of PFD
    // steps, which selects the prefetch slot and the buffer parity); false
    // ends this thread's steps (a wait ran out).  TAIL: the next steps, the
    // re-arm and the prefetch may lie past the end, so they are checked; the
    // main loop runs the steps where none can, without those checks.
    auto step = [&](auto P, auto TAIL, int s) -> bool {
        constexpr int p = decltype(P)::value;
        constexpr bool tail = decltype(TAIL)::value;
        const int par = p & 1;  // = s & 1: s0 is a multiple of the even PFD
        const int t = direction ? steps - 1 - s : s;
        // this step's projection values
        float gcur[NCH][HV];
        if constexpr (SRING) {
            ptx::cp_async_wait<GD - 1>();  // the copy issued GD steps ago
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
                for (int v = 0; v < HV; ++v)
                    gcur[ch][v] = gring[s & (GD - 1)][ch * HV + v][tid];
        } else {
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
                for (int v = 0; v < HV; ++v)
                    gcur[ch][v] = gq[p][ch][v];
        }

        if constexpr (CM) {
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
                // 0. this chunk's h_{s-1} complete in buffer `par`; then
                //    re-arm the barrier for h_{s+1}
                if (s > 0 && bar_bytes[ch] != 0) {
                    if (!wait_phase(&hbar[par][ch], ((s - 1) >> 1) & 1))
                        return false;
                    if (tid == 0 && (!tail || s + 2 < steps))
                        ptx::mbar_arrive_expect_tx(&hbar[par][ch], bar_bytes[ch]);
                }
                if constexpr (FLOOR) {
                    emit(par, ch, floor_h(par, ch, gcur[ch]), !tail || s + 1 < steps, t);
                } else {
                    float part[V], held[HV];
                    dots(par, ch, part);
                    reduce(part, held);
                    emit(par, ch, cell(ch, held, gcur[ch]), !tail || s + 1 < steps, t);
                }
            }
        } else {
            // 0. h_{s-1} complete in buffer `par`
            if (s > 0) {
                const uint32_t phase = ((s - 1) >> 1) & 1;
                volatile int *abort_v = &abort_flag;
                // A wait that runs out (or sees that another warp's did) ends
                // this thread's steps: it neither re-arms nor pushes again,
                // so no stuck barrier is armed or credited after the fault.
                if (!ptx::mbar_try_wait_cluster(&hbar[par][0], phase)) {
                    if (*abort_v)
                        return false;
                    const uint64_t start = ptx::globaltimer();
                    while (!ptx::mbar_try_wait_cluster(&hbar[par][0], phase)) {
                        if (*abort_v)
                            return false;
                        if (ptx::globaltimer() - start > wait_limit_ns) {
                            atomicOr(fault, kFaultRecurrence);
                            *abort_v = 1;
                            return false;
                        }
                    }
                }
                // re-arm this buffer for h_{s+1}
                if (tid == 0 && (!tail || s + 2 < steps))
                    ptx::mbar_arrive_expect_tx(&hbar[par][0], bar_bytes[0]);
            }

            float h[NCH];
            if constexpr (FLOOR) {
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch)
                    h[ch] = floor_h(par, ch, gcur[ch]);
            } else {
            // The chunks are independent: each phase below runs over all of
            // them, so their latencies overlap.
            // 1. partial dot products over this lane's K chunk
            float part[NCH][V];
    #pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
    #pragma unroll
                for (int w = 0; w < NW; ++w) {
                    const float4 *hp = reinterpret_cast<const float4 *>(
                        &hbuf[par][wbase + ch * NW + w][kc * CHUNK_STRIDE]);
                    const float4 h0 = hp[0], h1 = hp[1], h2 = hp[2], h3 = hp[3];
                    const float2 hh[8] = {{h0.x, h0.y}, {h0.z, h0.w}, {h1.x, h1.y},
                                          {h1.z, h1.w}, {h2.x, h2.y}, {h2.z, h2.w},
                                          {h3.x, h3.y}, {h3.z, h3.w}};
                    float2 acc[4];
    #pragma unroll
                    for (int q = 0; q < 4; ++q)
                        acc[q] = make_float2(0.0f, 0.0f);
    #pragma unroll
                    for (int i = 0; i < 8; ++i)
    #pragma unroll
                        for (int q = 0; q < 4; ++q)
                            acc[q] = __ffma2_rn(r2[q][i], hh[i], acc[q]);
    #pragma unroll
                    for (int q = 0; q < 4; ++q)
                        part[ch][w * 4 + q] = acc[q].x + acc[q].y;
                }
            }

            // 2. fixed butterfly over the 8 K-chunk lanes
            float held[NCH][HV];
    #pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
                if constexpr (V >= 8) {
                    float a[V / 2], b2[V / 4];
                    reduce_level<V, PERM>(part[ch], a, 4, (kc & 4) != 0);
                    reduce_level<V / 2, PERM>(a, b2, 2, (kc & 2) != 0);
                    reduce_level<V / 4, PERM>(b2, held[ch], 1, (kc & 1) != 0);
                } else {
                    float a[2], b2[1];
                    reduce_level<4, PERM>(part[ch], a, 4, (kc & 4) != 0);
                    reduce_level<2, PERM>(a, b2, 2, (kc & 2) != 0);
                    held[ch][0] = b2[0] + __shfl_xor_sync(0xffffffffu, b2[0], 1);
                }
            }

            // 3. activations, gate gather, cell update
    #pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
                float act[HV];
    #pragma unroll
                for (int v = 0; v < HV; ++v) {
                    const float w = held[ch][v] + fmaf(gcur[ch][v], gk[v], bias_v[v]);
                    act[v] = fmaf(act_m[v], inv_one_plus_ex2(w), act_a[v]);
                }
                float gate[4];
    #pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int src = V >= 8 ? (4 * wl + q) / HV : 2 * q;
                    gate[q] = __shfl_sync(0xffffffffu, act[q % HV], src, 8);
                }
                c[ch] = cell_update(gate[0], gate[1], gate[2], c[ch]);
                // h = o tanh(c) = o (2 r - 1) with r = 1 / (1 + 2^(-2 log2(e) c)):
                // one fused multiply-add after r
                const float r = inv_one_plus_ex2(c[ch] * (-2.0f * kLog2e));
                h[ch] = fmaf(2.0f * gate[3], r, -gate[3]);
            }

            }

            // 4. gather the warp's four units of window wl, push them (16
            //    bytes) into every CTA's next h buffer and store them to y
    #pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
                float h4[4];
    #pragma unroll
                for (int j = 0; j < 4; ++j)
                    h4[j] = __shfl_sync(0xffffffffu, h[ch], 8 * j + kc);
                if (bch0 + ch * NW + wl < batch) {
                    if (!tail || s + 1 < steps) {
                        const uint32_t off = static_cast<uint32_t>(ch * NW * HROW * 4);
    #pragma unroll
                        for (int r = 0; r < NPEER; ++r) {
                            if (sender + r * 4 * REPL < C)
                                ptx::st_async_v4(rdst[r][par ^ 1] + off, h4[0], h4[1], h4[2],
                                                 h4[3], rbar[r][par ^ 1]);
                        }
                    }
                    if (sender == 0)
                        *reinterpret_cast<float4 *>(ych0 + (ch * row_stride + t) * kOutput) =
                            make_float4(h4[0], h4[1], h4[2], h4[3]);
                }
            }
        }

        // 5. projection values PFD steps ahead
        if constexpr (SRING)
            gissue(s + GD);
        else
            gload(s + PFD, gq[p], tail);
        return true;
    };

    // Failure test: CTA 0 of the cluster pushes nothing, so its peers'
    // waits run out.
    if (withhold && rank == 0)
        goto done;
    {
        int s0 = 0;
        // every step of the group, its successor steps and its prefetch lie
        // before the end.  Measured (GB300, T = 589): 1-3 % faster per step
        // with 4 or 8 windows per chunk; with 1 or 2 it was up to 2 % slower,
        // so those run the checked loop only.
        if constexpr (NW >= 4) {
            for (; s0 + 2 * PFD <= steps; s0 += PFD)
                if (!unrolled_all<PFD>([&](auto P) {
                        return step(P, std::false_type{}, s0 + decltype(P)::value);
                    }))
                    goto done;
        }
        for (; s0 < steps; s0 += PFD)
            if (!unrolled_all<PFD>([&](auto P) {
                    const int s = s0 + decltype(P)::value;
                    return s < steps && step(P, std::true_type{}, s);
                }))
                break;
    }
done:
    if constexpr (SRING)
        ptx::cp_async_wait_all();  // no copy into this CTA's ring outlives it
    // no CTA leaves while a peer may still write into its shared memory
    __syncwarp();
    ptx::cluster_arrive_release();
    ptx::cluster_wait_acquire();
}

// Fused input projection (small batches): the recurrence computes its own
// projection values instead of reading G.  Clusters of 8 CTAs of 256 threads,
// one window per cluster.  Threads 0-127 run the recurrence exactly as the
// one-window kernel above (the same lanes, weights, butterfly and cell);
// threads 128-255 ("input lanes", one per recurrence lane: same unit, same
// K-chunk index kc) hold that lane's slice of the layer's input weights W
// (the 4 gate rows of the unit, columns kc*KIN/8 .. +KIN/8, W = hi + lo of
// the packed planes, scaled by the gates' k_q) and, running up to PD steps
// ahead, compute for every step the four partial sums of W x_t over their
// columns.  The recurrence lane adds them to its four partial sums of R h
// before the butterfly, so one reduction yields k_q (W x_t + R h) and the
// bias is added after it, as the projection value is in the unfused kernel.
// x_t reaches the CTA as one bulk copy per step (one input lane issues it XD
// steps ahead into a ring), and the partial sums reach the recurrence lanes
// through a shared-memory ring; every wait is bounded.  The products are fp32
// FMAs (the projection kernel's 3xTF32 form differs from it in the last bits).
template <int KIN>
__global__ void __launch_bounds__(256, 1)
recurrence_fused_kernel(const float *__restrict__ x, int in_width,
                        const float *__restrict__ wp_hi, const float *__restrict__ wp_lo,
                        const float *__restrict__ rp_in, const float *__restrict__ bias_in,
                        float *__restrict__ y, int batch, int steps, int dir_in,
                        unsigned *fault, unsigned long long wait_limit_ns, int withhold)
{
    constexpr int C = 8;
    constexpr int U = kHidden / C;  // 16 units per CTA
    constexpr int RT = 128;         // recurrence threads (and input threads)
    constexpr int KX = KIN / KC;    // input columns per lane
    constexpr int XD = 8;           // input-row ring slots
    constexpr int PD = 8;           // partial-sum ring slots
    // a row's K chunk kc (KX floats) sits at kc * XSTRIDE: the padding puts
    // the 8 lanes of a quarter-warp, which read the 8 chunks, in distinct banks
    constexpr int XSTRIDE = KX + 4;
    static_assert(KX % 4 == 0 && U * KC == RT, "fused shape");

    __shared__ __align__(16) float hbuf[2][HROW];
    __shared__ __align__(16) float xrow[XD][KC * XSTRIDE];
    __shared__ __align__(16) float4 xpart[PD][RT];
    __shared__ __align__(8) uint64_t hbar[2];
    __shared__ __align__(8) uint64_t xfull[XD], xempty[XD], pfull[PD], pempty[PD];
    __shared__ int abort_flag;

    const int tid = threadIdx.x;
    const bool input_lane = tid >= RT;
    const int lt = tid & (RT - 1);
    const int lane = tid & 31;
    const int kc = lt & 7;
    const int ul = lt >> 3;
    const uint32_t rank = ptx::cluster_ctarank();
    const int cid = static_cast<int>(ptx::cluster_id_x());
    const int direction = dir_in >= 0 ? dir_in : (cid & 1);
    const int win = dir_in >= 0 ? cid : (cid >> 1);  // this cluster's window
    const float *__restrict__ rp = rp_in + (dir_in >= 0 ? 0 : direction * kGates * kHidden);
    const float *__restrict__ bias = bias_in + (dir_in >= 0 ? 0 : direction * kGates);
    const int u = static_cast<int>(rank) * U + ul;
    const int u0 = u & ~3;
    // slot q of a lane's partial sums holds gate q ^ xq (the select-free
    // butterfly's lane-dependent order, as in the one-window kernel)
    const int xq = ((kc & 4) ? 2 : 0) | ((kc & 2) ? 1 : 0);
    volatile int *abort_v = &abort_flag;
    // The input lanes run ahead of the recurrence and mostly wait for a free
    // ring slot: they wait with a sleep between polls, so that they leave
    // the issue slots to the recurrence warps on the same SM sub-partitions.
    auto input_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        if (ptx::mbar_try_wait(bar, parity))
            return true;
        const uint64_t start = ptx::globaltimer();
        while (true) {
            __nanosleep(256);
            if (ptx::mbar_try_wait(bar, parity))
                return true;
            if (*abort_v)
                return false;
            if (ptx::globaltimer() - start > wait_limit_ns) {
                atomicOr(fault, kFaultRecurrence);
                *abort_v = 1;
                return false;
            }
        }
    };

    // weights: recurrence lanes R (columns kc*16 ..), input lanes W
    // (columns kc*KX ..), rows in slot order, scaled by k_q
    float2 r2[4][KLEN / 2];
    float2 w2[4][KX / 2];
    if (!input_lane) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int row = 4 * u + (q ^ xq);
            const float kq = (q ^ xq) == 2 ? -2.0f * kLog2e : -kLog2e;
            const float2 *src = reinterpret_cast<const float2 *>(rp + row * kHidden + kc * KLEN);
#pragma unroll
            for (int i = 0; i < KLEN / 2; ++i)
                r2[q][i] = make_float2(src[i].x * kq, src[i].y * kq);
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int row = direction * kGates + 4 * u + (q ^ xq);
            const float kq = (q ^ xq) == 2 ? -2.0f * kLog2e : -kLog2e;
            const float2 *hi = reinterpret_cast<const float2 *>(wp_hi + row * KIN + kc * KX);
            const float2 *lo = reinterpret_cast<const float2 *>(wp_lo + row * KIN + kc * KX);
#pragma unroll
            for (int i = 0; i < KX / 2; ++i)
                w2[q][i] = make_float2((hi[i].x + lo[i].x) * kq, (hi[i].y + lo[i].y) * kq);
        }
    }
    // after the reduction lane kc holds gate kc >> 1 (both lanes of a pair)
    const int gq = kc >> 1;
    const float gk = gq == 2 ? -2.0f * kLog2e : -kLog2e;
    const float bias_v = bias[4 * u + gq] * gk;
    const float act_m = gq == 2 ? 2.0f : 1.0f;
    const float act_a = gq == 2 ? -1.0f : 0.0f;

    for (int i = tid; i < 2 * HROW; i += 256)
        (&hbuf[0][0])[i] = 0.0f;
    for (int i = tid; i < XD * KC * XSTRIDE; i += 256)  // the padding stays zero
        (&xrow[0][0])[i] = 0.0f;
    ptx::fence_proxy_async_smem();  // before the bulk copies write the ring
    const uint32_t bar_bytes = kHidden * 4;  // one window
    if (tid == 0) {
        ptx::mbar_init(&hbar[0], 1);
        ptx::mbar_init(&hbar[1], 1);
        for (int i = 0; i < XD; ++i) {
            ptx::mbar_init(&xfull[i], 1);
            ptx::mbar_init(&xempty[i], RT / 32);
        }
        for (int i = 0; i < PD; ++i) {
            ptx::mbar_init(&pfull[i], RT / 32);
            ptx::mbar_init(&pempty[i], RT / 32);
        }
        abort_flag = 0;
        ptx::fence_mbar_init();
        if (steps > 1)
            ptx::mbar_arrive_expect_tx(&hbar[1], bar_bytes);
        if (steps > 2)
            ptx::mbar_arrive_expect_tx(&hbar[0], bar_bytes);
    }
    ptx::cluster_arrive_release();
    ptx::cluster_wait_acquire();
    ptx::griddep_launch_dependents();
    // launched as a programmatic dependent of the kernel that writes its
    // input: wait for that kernel's end before the first read of it
    ptx::griddep_wait();

    const uint32_t row_bytes = static_cast<uint32_t>(in_width) * 4;
    // step s's input row into ring slot `slot`, one bulk copy per K chunk
    // (the last chunk of a 60-wide row holds 4 columns; its rest stays zero)
    auto x_load = [&](int s, int slot) {
        const long t = direction ? steps - 1 - s : s;
        const float *src = x + (static_cast<long>(win) * steps + t) * in_width;
        ptx::mbar_arrive_expect_tx(&xfull[slot], row_bytes);
#pragma unroll
        for (int k = 0; k < KC; ++k) {
            const int cols = min(KX, in_width - k * KX);
            if (cols > 0)
                ptx::bulk_load(&xrow[slot][k * XSTRIDE], src + k * KX,
                               static_cast<uint32_t>(cols) * 4, &xfull[slot]);
        }
    };
    int x_issued = 0;  // input rows whose copies were issued (input lane 0)
    int x_done = 0;    // input rows consumed (every input lane)

    if (withhold && rank == 0)
        goto done;
    if (input_lane) {
        if (lt == 0)
            for (; x_issued < XD && x_issued < steps; ++x_issued)
                x_load(x_issued, x_issued);
        for (int s = 0; s < steps; ++s) {
            const int xs = s % XD, ps = s % PD;
            if (!input_wait(&xfull[xs], (s / XD) & 1))
                break;
            float2 acc[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                acc[q] = make_float2(0.0f, 0.0f);
            const float4 *xp = reinterpret_cast<const float4 *>(&xrow[xs][kc * XSTRIDE]);
#pragma unroll
            for (int i = 0; i < KX / 4; ++i) {
                const float4 v = xp[i];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[q] = __ffma2_rn(w2[q][2 * i], make_float2(v.x, v.y), acc[q]);
                    acc[q] = __ffma2_rn(w2[q][2 * i + 1], make_float2(v.z, v.w), acc[q]);
                }
            }
            x_done = s + 1;
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(&xempty[xs]);
            // the row XD steps on goes into this slot once every input lane
            // has read it
            if (lt == 0 && x_issued < steps) {
                if (!input_wait(&xempty[xs], (s / XD) & 1))
                    break;
                x_load(x_issued, xs);
                ++x_issued;
            }
            if (s >= PD && !input_wait(&pempty[ps], ((s / PD) - 1) & 1))
                break;
            xpart[ps][lt] = make_float4(acc[0].x + acc[0].y, acc[1].x + acc[1].y,
                                        acc[2].x + acc[2].y, acc[3].x + acc[3].y);
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(&pfull[ps]);
        }
        goto done;
    }
    {
        // the peers this lane sends its warp's four units to (lanes 0-7)
        const uint32_t hbase = ptx::smem_u32(&hbuf[0][0]);
        const uint32_t bar_base = ptx::smem_u32(&hbar[0]);
        const uint32_t send_off0 =
            static_cast<uint32_t>(((u0 / KLEN) * CHUNK_STRIDE + (u0 % KLEN)) * 4);
        const int peer = lane < C ? lane : C - 1;
        uint32_t rdst[2], rbar[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            rdst[q] = ptx::map_to_rank(hbase + static_cast<uint32_t>(q * HROW * 4) + send_off0,
                                       static_cast<uint32_t>(peer));
            rbar[q] = ptx::map_to_rank(bar_base + static_cast<uint32_t>(q * 8),
                                       static_cast<uint32_t>(peer));
        }
        float *yrow = y + static_cast<long>(win) * steps * kOutput + direction * kHidden + u0;
        float c = 0.0f;
        for (int s = 0; s < steps; ++s) {
            const int par = s & 1, ps = s % PD;
            const int t = direction ? steps - 1 - s : s;
            // this step's input partial sums (normally long ready)
            if (!ptx::mbar_wait_bounded(&pfull[ps], (s / PD) & 1, abort_v, fault,
                                        kFaultRecurrence, wait_limit_ns))
                break;
            const float4 xs4 = xpart[ps][lt];
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(&pempty[ps]);
            // h_{s-1} complete in buffer par; re-arm it for h_{s+1}
            if (s > 0) {
                const uint32_t phase = ((s - 1) >> 1) & 1;
                if (!ptx::mbar_try_wait_cluster(&hbar[par], phase)) {
                    if (*abort_v)
                        break;
                    const uint64_t start = ptx::globaltimer();
                    bool ok = true;
                    while (!ptx::mbar_try_wait_cluster(&hbar[par], phase)) {
                        if (*abort_v || ptx::globaltimer() - start > wait_limit_ns) {
                            if (!*abort_v) {
                                atomicOr(fault, kFaultRecurrence);
                                *abort_v = 1;
                            }
                            ok = false;
                            break;
                        }
                    }
                    if (!ok)
                        break;
                }
                if (tid == 0 && s + 2 < steps)
                    ptx::mbar_arrive_expect_tx(&hbar[par], bar_bytes);
            }
            // R h over this lane's K chunk, plus W x_t of the input lane
            const float4 *hp = reinterpret_cast<const float4 *>(&hbuf[par][kc * CHUNK_STRIDE]);
            const float4 h0 = hp[0], h1 = hp[1], h2 = hp[2], h3 = hp[3];
            const float2 hh[8] = {{h0.x, h0.y}, {h0.z, h0.w}, {h1.x, h1.y}, {h1.z, h1.w},
                                  {h2.x, h2.y}, {h2.z, h2.w}, {h3.x, h3.y}, {h3.z, h3.w}};
            const float xs[4] = {xs4.x, xs4.y, xs4.z, xs4.w};
            float part[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    acc = __ffma2_rn(r2[q][i], hh[i], acc);
                part[q] = (acc.x + acc.y) + xs[q];
            }
            float a[2], b2[1];
            reduce_level<4, true>(part, a, 4, (kc & 4) != 0);
            reduce_level<2, true>(a, b2, 2, (kc & 2) != 0);
            const float held = b2[0] + __shfl_xor_sync(0xffffffffu, b2[0], 1);
            const float act = fmaf(act_m, inv_one_plus_ex2(held + bias_v), act_a);
            float gate[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                gate[q] = __shfl_sync(0xffffffffu, act, 2 * q, 8);
            c = cell_update(gate[0], gate[1], gate[2], c);
            const float r = inv_one_plus_ex2(c * (-2.0f * kLog2e));
            const float h = fmaf(2.0f * gate[3], r, -gate[3]);
            float h4[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                h4[j] = __shfl_sync(0xffffffffu, h, 8 * j + kc);
            if (s + 1 < steps && lane < C)
                ptx::st_async_v4(rdst[par ^ 1], h4[0], h4[1], h4[2], h4[3], rbar[par ^ 1]);
            if (lane == 0)
                *reinterpret_cast<float4 *>(yrow + static_cast<long>(t) * kOutput) =
                    make_float4(h4[0], h4[1], h4[2], h4[3]);
        }
    }
done:
    if (input_lane && lt == 0) {
        // every issued input row has landed before the shared memory goes away
        for (int s = x_done; s < x_issued; ++s)
            ptx::mbar_wait_drain(&xfull[s % XD], (s / XD) & 1, fault, kDefaultWaitLimitNs);
    }
    __syncwarp();
    ptx::cluster_arrive_release();
    ptx::cluster_wait_acquire();
}

// Two units per 8-lane group (one window per cluster, clusters of 8 CTAs of
// 64 threads): lane kc of group g holds the R slices of two hidden units,
// base + g and base + 4 + g (base = the warp's first of 8 units), for K chunk
// kc, loads its h chunk once and multiplies it into 8 gate rows.  Against one
// unit per group this halves the shared-memory loads of h per step (every
// 128-bit load costs the load/store unit four cycles however many lanes
// read the same address) and the warps per SM, for twice the FFMA2 chains per
// lane.  The partial sums of the two units are reduced like two windows of
// the two-window variants (the same 8-value butterfly, select-free: lane kc
// keeps its partial sums in the order p -> p ^ kc, which here only changes
// which unit and gate row a register slot holds, since every slot reads the
// same h), so each unit's z is the sum of the same eight chunk partials in the
// same order as in every other variant: results are bitwise identical.
template <bool FLOOR = false, int C = 8>
__global__ void __launch_bounds__(512 / C, 1)
recurrence_u2_kernel(const float *__restrict__ g, const float *__restrict__ rp_in,
                     const float *__restrict__ bias_in, float *__restrict__ y, int batch, int steps,
                     int dir_in, unsigned *fault, unsigned long long wait_limit_ns, int withhold)
{
    static_assert(C == 4 || C == 8, "cluster");
    constexpr int THREADS = 512 / C;  // the CTA's 128 / C units, two per lane group
    constexpr int GD = 64;  // projection-value ring depth (steps)

    __shared__ __align__(16) float hbuf[2][HROW];
    __shared__ __align__(8) uint64_t hbar[2];
    __shared__ int abort_flag;
    __shared__ __align__(16) float gring[GD][THREADS];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int kc = tid & 7;
    const int grp = (tid >> 3) & 3;
    const int jj = kc >> 2;                    // after the reduction: unit index 0/1
    const int q = kc & 3;                      // and gate
    const uint32_t rank = ptx::cluster_ctarank();
    const int cid = static_cast<int>(ptx::cluster_id_x());
    const int direction = dir_in >= 0 ? dir_in : (cid & 1);
    const int win = dir_in >= 0 ? cid : (cid >> 1);
    const float *__restrict__ rp = rp_in + (dir_in >= 0 ? 0 : direction * kGates * kHidden);
    const float *__restrict__ bias = bias_in + (dir_in >= 0 ? 0 : direction * kGates);
    const int base = static_cast<int>(rank) * (kHidden / C) + (tid >> 5) * 8;  // the warp's 8 units
    volatile int *abort_v = &abort_flag;

    // R slices of the group's two units for chunk kc, scaled by k_q; slot
    // (j, gq) holds unit index j ^ (kc >> 2), gate gq ^ (kc & 3)
    float2 r2[2][4][KLEN / 2];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int gq = 0; gq < 4; ++gq) {
            const int jl = j ^ (kc >> 2), ql = gq ^ (kc & 3);
            const int row = 4 * (base + 4 * jl + grp) + ql;
            const float kq = ql == 2 ? -2.0f * kLog2e : -kLog2e;
            const float2 *src = reinterpret_cast<const float2 *>(rp + row * kHidden + kc * KLEN);
#pragma unroll
            for (int i = 0; i < KLEN / 2; ++i)
                r2[j][gq][i] = make_float2(src[i].x * kq, src[i].y * kq);
        }
    // the value this lane holds after the reduction: unit base + 4 jj + grp, gate q
    const int u_mine = base + 4 * jj + grp;
    const float gk = q == 2 ? -2.0f * kLog2e : -kLog2e;
    const float bias_v = bias[4 * u_mine + q] * gk;
    const float act_m = q == 2 ? 2.0f : 1.0f;
    const float act_a = q == 2 ? -1.0f : 0.0f;
    const float *gcol = g + direction * kGates + 4 * u_mine + q +
                        static_cast<long>(win) * steps * kGateColumns;

    for (int i = tid; i < 2 * HROW; i += THREADS)
        (&hbuf[0][0])[i] = 0.0f;
    const uint32_t bar_bytes = kHidden * 4;
    if (tid == 0) {
        ptx::mbar_init(&hbar[0], 1);
        ptx::mbar_init(&hbar[1], 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
        if (steps > 1)
            ptx::mbar_arrive_expect_tx(&hbar[1], bar_bytes);
        if (steps > 2)
            ptx::mbar_arrive_expect_tx(&hbar[0], bar_bytes);
    }
    ptx::cluster_arrive_release();
    ptx::cluster_wait_acquire();
    ptx::griddep_launch_dependents();
    // launched as a programmatic dependent of the kernel that writes its
    // input: wait for that kernel's end before the first read of it
    ptx::griddep_wait();

    // senders: lane group*4 + kc%4 (< 8) pushes units base + 4 jj .. +3 to
    // that peer; lanes kc = 0 and 4 of group 0 store them to y
    const int sender = grp * 4 + (kc & 3);
    const int u4 = base + 4 * jj;  // first of the four units this lane gathers
    const uint32_t hbase = ptx::smem_u32(&hbuf[0][0]);
    const uint32_t bar_base = ptx::smem_u32(&hbar[0]);
    const uint32_t send_off =
        static_cast<uint32_t>(((u4 / KLEN) * CHUNK_STRIDE + (u4 % KLEN)) * 4);
    const int peer = sender < C ? sender : C - 1;
    uint32_t rdst[2], rbar[2];
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        rdst[b] = ptx::map_to_rank(hbase + static_cast<uint32_t>(b * HROW * 4) + send_off,
                                   static_cast<uint32_t>(peer));
        rbar[b] = ptx::map_to_rank(bar_base + static_cast<uint32_t>(b * 8),
                                   static_cast<uint32_t>(peer));
    }
    float *yrow = y + static_cast<long>(win) * steps * kOutput + direction * kHidden + u4;

    auto gissue = [&](int s) {
        const long t = direction ? steps - 1 - s : s;
        const bool ok = s < steps;
        ptx::cp_async_4(ptx::smem_u32(&gring[s & (GD - 1)][tid]),
                        ok ? gcol + t * kGateColumns : g, ok ? 4u : 0u);
        ptx::cp_async_commit();
    };
    for (int s = 0; s < GD; ++s)
        gissue(s);

    float c = 0.0f;
    auto step = [&](auto PAR, int s) -> bool {
        constexpr int par = decltype(PAR)::value;
        const int t = direction ? steps - 1 - s : s;
        ptx::cp_async_wait<GD - 1>();
        const float gv = gring[s & (GD - 1)][tid];
        if (s > 0) {
            const uint32_t phase = ((s - 1) >> 1) & 1;
            if (!ptx::mbar_try_wait_cluster(&hbar[par], phase)) {
                if (*abort_v)
                    return false;
                const uint64_t start = ptx::globaltimer();
                while (!ptx::mbar_try_wait_cluster(&hbar[par], phase)) {
                    if (*abort_v)
                        return false;
                    if (ptx::globaltimer() - start > wait_limit_ns) {
                        atomicOr(fault, kFaultRecurrence);
                        *abort_v = 1;
                        return false;
                    }
                }
            }
            if (tid == 0 && s + 2 < steps)
                ptx::mbar_arrive_expect_tx(&hbar[par], bar_bytes);
        }
        float h;
        if constexpr (FLOOR) {
            h = fmaf(hbuf[par][kc * CHUNK_STRIDE], 0.5f, gv * 0.001f);
        } else {
            const float4 *hp = reinterpret_cast<const float4 *>(&hbuf[par][kc * CHUNK_STRIDE]);
            const float4 h0 = hp[0], h1 = hp[1], h2 = hp[2], h3 = hp[3];
            const float2 hh[8] = {{h0.x, h0.y}, {h0.z, h0.w}, {h1.x, h1.y}, {h1.z, h1.w},
                                  {h2.x, h2.y}, {h2.z, h2.w}, {h3.x, h3.y}, {h3.z, h3.w}};
            // the eight rows' chains advance together; each chain's order
            // over i is fixed
            float2 acc[8];
#pragma unroll
            for (int r = 0; r < 8; ++r)
                acc[r] = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    acc[r] = __ffma2_rn(r2[r >> 2][r & 3][i], hh[i], acc[r]);
            float part[8];
#pragma unroll
            for (int r = 0; r < 8; ++r)
                part[r] = acc[r].x + acc[r].y;
            float a[4], b2[2], held[1];
            reduce_level<8, true>(part, a, 4, (kc & 4) != 0);
            reduce_level<4, true>(a, b2, 2, (kc & 2) != 0);
            reduce_level<2, true>(b2, held, 1, (kc & 1) != 0);
            const float w = held[0] + fmaf(gv, gk, bias_v);
            const float act = fmaf(act_m, inv_one_plus_ex2(w), act_a);
            float gate[4];
#pragma unroll
            for (int gq = 0; gq < 4; ++gq)
                gate[gq] = __shfl_sync(0xffffffffu, act, 4 * jj + gq, 8);
            c = cell_update(gate[0], gate[1], gate[2], c);
            const float r = inv_one_plus_ex2(c * (-2.0f * kLog2e));
            h = fmaf(2.0f * gate[3], r, -gate[3]);
        }
        float h4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            h4[k] = __shfl_sync(0xffffffffu, h, 8 * k + kc);
        if (s + 1 < steps && sender < C)
            ptx::st_async_v4(rdst[par ^ 1], h4[0], h4[1], h4[2], h4[3], rbar[par ^ 1]);
        if (sender == 0 && lane < 8)
            *reinterpret_cast<float4 *>(yrow + static_cast<long>(t) * kOutput) =
                make_float4(h4[0], h4[1], h4[2], h4[3]);
        gissue(s + GD);
        return true;
    };

    if (withhold && rank == 0)
        goto done;
    for (int s0 = 0; s0 < steps; s0 += 2) {
        if (!step(std::integral_constant<int, 0>{}, s0))
            break;
        if (s0 + 1 < steps && !step(std::integral_constant<int, 1>{}, s0 + 1))
            break;
    }
done:
    ptx::cp_async_wait_all();
    __syncwarp();
    ptx::cluster_arrive_release();
    ptx::cluster_wait_acquire();
}

// Two units per 8-lane group for several windows per lane: NW = 4 or 8
// windows per chunk, NCH = 1 or 2 chunks, clusters of C = 4 or 8 CTAs of
// 512 / C threads (a CTA's 128 / C units, two per group).  Lane kc of group g
// holds the R slices of units base + g and base + 4 + g (base = the warp's
// first of 8 units) for K chunk kc and multiplies each window's h chunk into
// their 8 gate rows: half the shared-memory loads of h per multiply-add of
// the one-unit variants.  The select-free butterfly keeps a chunk's partial
// sums in the order L -> L ^ (NW kc), L = 8 w + 4 j + q (window w, unit j,
// gate q), so the three levels leave lane kc the four gates of whole cells
// (window kc / 2 of unit kc % 2 for NW = 4; both units of window kc for
// NW = 8) and the cell update needs no gate gather.  The order only permutes
// which unit a register slot holds and which window row a slot reads (the
// senders store window w of K chunk k at row w ^ (NW k / 8)): every unit's z
// is the same sums in the same order as in every other variant, so results
// are bitwise identical.  Two chunks run chunk-major with a barrier pair
// each, so one chunk's exchange is in flight while the other computes.
template <int C, int NW, int NCH, bool FLOOR = false>
__global__ void __launch_bounds__(512 / C, 1)
recurrence_u2w_kernel(const float *__restrict__ g, const float *__restrict__ rp_in,
                      const float *__restrict__ bias_in, float *__restrict__ y, int batch,
                      int steps, int dir_in, unsigned *fault, unsigned long long wait_limit_ns,
                      int withhold)
{
    constexpr int THREADS = 512 / C;
    constexpr int UPC = kHidden / C;  // units per CTA
    constexpr int TW = NW * NCH;      // windows per cluster
    constexpr int V = 8 * NW;         // partial sums per lane and chunk
    constexpr int HV = V / 8;         // values a lane holds after the reduction
    // cells a lane updates per chunk; with two windows a lane holds two of
    // a cell's four gates and completes the cell with its partner lane kc ^ 1
    constexpr int CELLS = HV >= 4 ? HV / 4 : 1;
    // peers each holder of an h quad sends to (with C = 2 only the first two
    // of its four holders send)
    constexpr int NPEER = C >= 4 ? C / 4 : 1;
    constexpr bool CM = NCH > 1;
    constexpr int NBAR = CM ? NCH : 1;
    static_assert((C == 2 || C == 4 || C == 8) && (NW == 2 || NW == 4 || NW == 8) &&
                      (NCH == 1 || NCH == 2),
                  "shape");
    // projection values: a ring of GD steps in shared memory, each lane's
    // four gate values of a cell one 16-byte asynchronous copy
    constexpr int GD_FIT = (45056 - 2 * TW * HROW * 4) / (NCH * CELLS * THREADS * 16);
    static_assert(GD_FIT >= 4, "ring");
    constexpr int GD = GD_FIT >= 32 ? 32 : GD_FIT >= 16 ? 16 : GD_FIT >= 8 ? 8 : 4;
    constexpr float K0 = -kLog2e, K2 = -2.0f * kLog2e;  // k_q of the gates, the candidate

    __shared__ __align__(16) float hbuf[2][TW][HROW];
    __shared__ __align__(8) uint64_t hbar[2][NBAR];
    __shared__ int abort_flag;
    __shared__ __align__(16) float4 gring[GD][NCH * CELLS][THREADS];

    const int tid = threadIdx.x;
    const int kc = tid & 7;
    const int grp = (tid >> 3) & 3;
    const uint32_t rank = ptx::cluster_ctarank();
    const int cid = static_cast<int>(ptx::cluster_id_x());
    const int direction = dir_in >= 0 ? dir_in : (cid & 1);
    const int tile = dir_in >= 0 ? cid : (cid >> 1);
    const float *__restrict__ rp = rp_in + (dir_in >= 0 ? 0 : direction * kGates * kHidden);
    const float *__restrict__ bias = bias_in + (dir_in >= 0 ? 0 : direction * kGates);
    const int base = static_cast<int>(rank) * UPC + (tid >> 5) * 8;  // the warp's 8 units
    const int tile_w0 = tile * TW;
    volatile int *abort_v = &abort_flag;
    // window, unit and gate parts of the lane order L -> L ^ (HV k) of K chunk k
    auto xw = [](int k) { return (HV * k) >> 3; };
    auto xj = [](int k) { return ((HV * k) >> 2) & 1; };
    auto xq = [](int k) { return (HV * k) & 3; };

    // R slices: slot (js, q) holds gate q ^ xq(kc) of unit index js ^ xj(kc),
    // scaled by k_q
    float2 r2[2][4][KLEN / 2];
#pragma unroll
    for (int js = 0; js < 2; ++js)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int ql = q ^ xq(kc);
            const int row = 4 * (base + 4 * (js ^ xj(kc)) + grp) + ql;
            const float kq = ql == 2 ? K2 : K0;
            const float2 *src = reinterpret_cast<const float2 *>(rp + row * kHidden + kc * KLEN);
#pragma unroll
            for (int i = 0; i < KLEN / 2; ++i)
                r2[js][q][i] = make_float2(src[i].x * kq, src[i].y * kq);
        }

    // the cells this lane updates: logical values HV kc + 4 ci .. + 3
    int wc[CELLS];
    float bias_v[CELLS][4];
    const float *gsrc[CELLS];
    uint32_t send_off[CELLS];
    int u4c[CELLS];
#pragma unroll
    for (int ci = 0; ci < CELLS; ++ci) {
        const int l = HV * kc + 4 * ci;
        wc[ci] = l >> 3;
        const int jc = (l >> 2) & 1;
        const int u = base + 4 * jc + grp;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            bias_v[ci][q] = bias[4 * u + q] * (q == 2 ? K2 : K0);
        gsrc[ci] = g + direction * kGates + 4 * u +
                   static_cast<long>(tile_w0 + wc[ci]) * steps * kGateColumns;
        // after the h gather: units u4 .. u4 + 3 of window wc, in K chunk u4 / 16
        const int u4 = base + 4 * jc;
        u4c[ci] = u4;
        const int k = u4 / KLEN;
        send_off[ci] = static_cast<uint32_t>(
            ((wc[ci] ^ xw(k)) * HROW + k * CHUNK_STRIDE + (u4 % KLEN)) * 4);
    }

    uint32_t bar_bytes[NBAR];
#pragma unroll
    for (int b = 0; b < NBAR; ++b) {
        const int w0 = tile_w0 + (CM ? b * NW : 0);
        bar_bytes[b] = static_cast<uint32_t>(kHidden * 4 * max(0, min(CM ? NW : TW, batch - w0)));
    }

    for (int i = tid; i < 2 * TW * HROW; i += THREADS)
        (&hbuf[0][0][0])[i] = 0.0f;
    if (tid == 0) {
        for (int b = 0; b < NBAR; ++b) {
            ptx::mbar_init(&hbar[0][b], 1);
            ptx::mbar_init(&hbar[1][b], 1);
        }
        abort_flag = 0;
        ptx::fence_mbar_init();
        // a chunk with no window inside the batch has no barrier traffic
        for (int b = 0; b < NBAR; ++b) {
            if (bar_bytes[b] == 0)
                continue;
            if (steps > 1)
                ptx::mbar_arrive_expect_tx(&hbar[1][b], bar_bytes[b]);
            if (steps > 2)
                ptx::mbar_arrive_expect_tx(&hbar[0][b], bar_bytes[b]);
        }
    }
    ptx::cluster_arrive_release();
    ptx::cluster_wait_acquire();
    ptx::griddep_launch_dependents();
    // launched as a programmatic dependent of the kernel that writes its
    // input: wait for that kernel's end before the first read of it
    ptx::griddep_wait();

    // this lane's pushes: the four holders of an h quad (one per group)
    // send to peers grp, grp + 4 (C = 8) or grp (C = 4)
    const uint32_t hbase = ptx::smem_u32(&hbuf[0][0][0]);
    const uint32_t bar_base = ptx::smem_u32(&hbar[0][0]);
    uint32_t rdst[CELLS][NPEER][2], rbar[NPEER][2];
#pragma unroll
    for (int r = 0; r < NPEER; ++r) {
        const uint32_t peer = static_cast<uint32_t>(min(grp + 4 * r, C - 1));
#pragma unroll
        for (int b = 0; b < 2; ++b) {
#pragma unroll
            for (int ci = 0; ci < CELLS; ++ci)
                rdst[ci][r][b] = ptx::map_to_rank(
                    hbase + static_cast<uint32_t>(b * TW * HROW * 4) + send_off[ci], peer);
            rbar[r][b] = ptx::map_to_rank(bar_base + static_cast<uint32_t>(b * NBAR * 8), peer);
        }
    }

    auto valid = [&](int ch, int ci) { return tile_w0 + ch * NW + wc[ci] < batch; };
    auto gissue = [&](int s) {
        const long t = direction ? steps - 1 - s : s;
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
            for (int ci = 0; ci < CELLS; ++ci) {
                const bool ok = s < steps && valid(ch, ci);
                const float *src =
                    ok ? gsrc[ci] + (static_cast<long>(ch) * NW * steps + t) * kGateColumns : g;
                ptx::cp_async_16(ptx::smem_u32(&gring[s & (GD - 1)][ch * CELLS + ci][tid]), src,
                                 ok ? 16u : 0u);
            }
        ptx::cp_async_commit();
    };
    for (int s = 0; s < GD; ++s)
        gissue(s);

    float c[NCH][CELLS];
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
        for (int ci = 0; ci < CELLS; ++ci)
            c[ch][ci] = 0.0f;

    // waits until phase `phase` of `bar` completes; false if the wait ran out
    // here or in another warp (this thread then neither re-arms nor pushes)
    auto wait_phase = [&](uint64_t *bar, uint32_t phase) -> bool {
        if (ptx::mbar_try_wait_cluster(bar, phase))
            return true;
        if (*abort_v)
            return false;
        const uint64_t start = ptx::globaltimer();
        while (!ptx::mbar_try_wait_cluster(bar, phase)) {
            if (*abort_v)
                return false;
            if (ptx::globaltimer() - start > wait_limit_ns) {
                atomicOr(fault, kFaultRecurrence);
                *abort_v = 1;
                return false;
            }
        }
        return true;
    };

    auto step = [&](auto PAR, int s) -> bool {
        constexpr int par = decltype(PAR)::value;
        const int t = direction ? steps - 1 - s : s;
        const bool push = s + 1 < steps;
        ptx::cp_async_wait<GD - 1>();
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
            // this chunk's h_{s-1} complete in buffer `par` (a chunk past the
            // batch has no traffic); then re-arm the barrier for h_{s+1}
            if (s > 0 && bar_bytes[ch] != 0) {
                if (!wait_phase(&hbar[par][ch], ((s - 1) >> 1) & 1))
                    return false;
                if (tid == 0 && s + 2 < steps)
                    ptx::mbar_arrive_expect_tx(&hbar[par][ch], bar_bytes[ch]);
            }
            float h[CELLS];
            if constexpr (FLOOR) {
#pragma unroll
                for (int ci = 0; ci < CELLS; ++ci) {
                    const float4 gv = gring[s & (GD - 1)][ch * CELLS + ci][tid];
                    h[ci] = fmaf(hbuf[par][ch * NW][kc * CHUNK_STRIDE], 0.5f, gv.x * 0.001f);
                }
            } else {
                float part[V];
#pragma unroll
                for (int ws = 0; ws < NW; ++ws) {
                    const float4 *hp =
                        reinterpret_cast<const float4 *>(&hbuf[par][ch * NW + ws][kc * CHUNK_STRIDE]);
                    const float4 h0 = hp[0], h1 = hp[1], h2 = hp[2], h3 = hp[3];
                    const float2 hh[8] = {{h0.x, h0.y}, {h0.z, h0.w}, {h1.x, h1.y},
                                          {h1.z, h1.w}, {h2.x, h2.y}, {h2.z, h2.w},
                                          {h3.x, h3.y}, {h3.z, h3.w}};
                    // the eight rows' chains advance together; each
                    // chain's order over i is fixed
                    float2 acc[8];
#pragma unroll
                    for (int r = 0; r < 8; ++r)
                        acc[r] = make_float2(0.0f, 0.0f);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
#pragma unroll
                        for (int r = 0; r < 8; ++r)
                            acc[r] = __ffma2_rn(r2[r >> 2][r & 3][i], hh[i], acc[r]);
#pragma unroll
                    for (int r = 0; r < 8; ++r)
                        part[ws * 8 + r] = acc[r].x + acc[r].y;
                }
                float a[V / 2], b2[V / 4], held[V / 8];
                reduce_level<V, true>(part, a, 4, (kc & 4) != 0);
                reduce_level<V / 2, true>(a, b2, 2, (kc & 2) != 0);
                reduce_level<V / 4, true>(b2, held, 1, (kc & 1) != 0);
                if constexpr (NW == 2) {
                    // held[i]: gate 2 qh + i of this lane's cell (qh = kc & 1);
                    // lane kc ^ 1 holds the other two: swap the activated pair
                    const float4 gv = gring[s & (GD - 1)][ch][tid];
                    const bool qh = (kc & 1) != 0;
                    const float w0 = held[0] + fmaf(qh ? gv.z : gv.x, qh ? K2 : K0,
                                                    qh ? bias_v[0][2] : bias_v[0][0]);
                    const float w1 = held[1] + fmaf(qh ? gv.w : gv.y, K0,
                                                    qh ? bias_v[0][3] : bias_v[0][1]);
                    const float a0 =
                        fmaf(qh ? 2.0f : 1.0f, inv_one_plus_ex2(w0), qh ? -1.0f : 0.0f);
                    const float a1 = inv_one_plus_ex2(w1);
                    const float o0 = __shfl_xor_sync(0xffffffffu, a0, 1);
                    const float o1 = __shfl_xor_sync(0xffffffffu, a1, 1);
                    const float gi = qh ? o0 : a0, gf = qh ? o1 : a1;
                    const float gg = qh ? a0 : o0, go = qh ? a1 : o1;
                    c[ch][0] = cell_update(gi, gf, gg, c[ch][0]);
                    const float r = inv_one_plus_ex2(c[ch][0] * (-2.0f * kLog2e));
                    h[0] = fmaf(2.0f * go, r, -go);
                } else {
#pragma unroll
                for (int ci = 0; ci < CELLS; ++ci) {
                    const float4 gv = gring[s & (GD - 1)][ch * CELLS + ci][tid];
                    const float gq[4] = {gv.x, gv.y, gv.z, gv.w};
                    float act[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float w =
                            held[4 * ci + q] + fmaf(gq[q], q == 2 ? K2 : K0, bias_v[ci][q]);
                        act[q] = q == 2 ? fmaf(2.0f, inv_one_plus_ex2(w), -1.0f)
                                        : fmaf(1.0f, inv_one_plus_ex2(w), 0.0f);
                    }
                    c[ch][ci] = cell_update(act[0], act[1], act[2], c[ch][ci]);
                    const float r = inv_one_plus_ex2(c[ch][ci] * (-2.0f * kLog2e));
                    h[ci] = fmaf(2.0f * act[3], r, -act[3]);
                }
                }
            }
            // gather the group's four units of each cell's window, push the
            // quad to the peers, store it to y
#pragma unroll
            for (int ci = 0; ci < CELLS; ++ci) {
                float h4[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    h4[k] = __shfl_sync(0xffffffffu, h[ci], 8 * k + kc);
                // with two windows the pair kc, kc ^ 1 holds the same cell:
                // the even lane sends and stores it
                if (valid(ch, ci) && (NW != 2 || (kc & 1) == 0)) {
                    if (push) {
                        const uint32_t off = static_cast<uint32_t>(ch * NW * HROW * 4);
                        const uint32_t bar_off = static_cast<uint32_t>(CM ? ch * 8 : 0);
#pragma unroll
                        for (int r = 0; r < NPEER; ++r)
                            if (C >= 4 || grp < C)
                                ptx::st_async_v4(rdst[ci][r][par ^ 1] + off, h4[0], h4[1],
                                                 h4[2], h4[3], rbar[r][par ^ 1] + bar_off);
                    }
                    if (grp == 0)
                        *reinterpret_cast<float4 *>(
                            y + (static_cast<long>(tile_w0 + ch * NW + wc[ci]) * steps + t) * kOutput +
                            direction * kHidden + u4c[ci]) = make_float4(h4[0], h4[1], h4[2], h4[3]);
                }
            }
        }
        gissue(s + GD);
        return true;
    };

    if (withhold && rank == 0)
        goto done;
    for (int s0 = 0; s0 < steps; s0 += 2) {
        if (!step(std::integral_constant<int, 0>{}, s0))
            break;
        if (s0 + 1 < steps && !step(std::integral_constant<int, 1>{}, s0 + 1))
            break;
    }
done:
    ptx::cp_async_wait_all();
    __syncwarp();
    ptx::cluster_arrive_release();
    ptx::cluster_wait_acquire();
}

// Tensor-core recurrence for large batches: one cluster of 4 CTAs of 128
// threads per (direction, tile of 16 windows).  CTA rank r owns units
// [32 r, 32 r + 32): 128 gate rows, row m = 32 q + u for gate q of unit
// 32 r + u.  Its R rows, scaled by k_q and split into TF32 hi and lo parts,
// stay in tensor memory for the whole kernel as the MMAs' A operand
// (columns 0-127 hi, 128-255 lo).  Each step
//     z (128 rows x 16 windows, tensor memory) = A_hi.h_hi + A_hi.h_lo + A_lo.h_hi
// over K = 128: 48 tcgen05.mma kind::tf32 (M = 128, N = 16, K = 8) issued by
// one thread, with h (16 windows x 128 units, the B operand) in shared memory
// as TF32 hi and lo planes in the 64-byte-swizzled K-major layout.  Then warp
// q copies the z of gate q (its 32 tensor-memory lanes) into shared memory,
// and each thread updates 4 cells (window tid / 8, units 4 (tid % 8) .. + 3)
// with its prefetched projection values and the bias, stores h to y and,
// split into hi and lo, into its CTA's slice of the next step's B buffer;
// one thread then copies that 4 KiB slice into the same place of the three
// peer CTAs (cp.async.bulk shared::cta -> shared::cluster, credited to their
// mbarrier).  Padding windows past the batch are computed on zero projection
// values (each window's column of z depends on its own row of h only) and
// never stored.  The sums run in another order than the FFMA variants', so
// results agree with theirs to rounding, not bitwise.
constexpr int TC_N = 16;                           // windows per tile
constexpr int TC_C = 4;                            // CTAs per cluster
constexpr int TC_THREADS = 128;
constexpr int TC_GD = 4;                           // projection-value ring depth (steps)
constexpr int TC_KB_BYTES = TC_N * 64;             // one 16-column K-block of one plane
constexpr int TC_SLICE_BYTES = 2 * 2 * TC_KB_BYTES;  // a CTA's 32 units: 2 planes x 2 K-blocks
constexpr int TC_B_BYTES = TC_C * TC_SLICE_BYTES;    // one step's h
constexpr int TC_OFF_Z = 2 * TC_B_BYTES;             // after the two B buffers
constexpr int TC_Z_BYTES = 4 * TC_N * 32 * 4;        // z of 4 gates x 16 windows x 32 units
constexpr int TC_OFF_G = TC_OFF_Z + TC_Z_BYTES;
constexpr int TC_G_BYTES = TC_GD * TC_THREADS * 16 * 4;  // 16 projection values per thread
constexpr int TC_OFF_BAR = TC_OFF_G + TC_G_BYTES;
// More than half of an SM's shared memory, so one CTA per SM: each holds all
// 512 tensor-memory columns, and a second CTA on the SM would wait in its
// allocation for the first to end.
constexpr int TC_SMEM = 120 * 1024 + 1024;
constexpr uint32_t TC_AHI = 0, TC_ALO = 128, TC_D = 256, TC_TMEM_COLS = 512;
constexpr uint32_t TC_IDESC = ptx::tf32_idesc(128, TC_N);
static_assert(TC_OFF_BAR + 64 + 1024 <= TC_SMEM, "tensor-core recurrence shared memory");

template <bool FLOOR = false>
__global__ void __launch_bounds__(TC_THREADS, 1)
recurrence_tc_kernel(const float *__restrict__ g, const float *__restrict__ rp_in,
                     const float *__restrict__ bias_in, float *__restrict__ y, int batch,
                     int steps, int dir_in, unsigned *fault, unsigned long long wait_limit_ns,
                     int withhold)
{
    constexpr float K0 = -kLog2e, K2 = -2.0f * kLog2e;  // k_q of the gates, the candidate
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *hfull = reinterpret_cast<uint64_t *>(smem + TC_OFF_BAR);  // [2]: peers' slices
    uint64_t *mma_bar = hfull + 2;    // this step's MMAs complete
    uint64_t *drain_bar = hfull + 3;  // every MMA issued complete (teardown)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(hfull + 4);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *zbuf = reinterpret_cast<float *>(smem + TC_OFF_Z);   // [4 gates][16 windows][32 units]
    float *gring = reinterpret_cast<float *>(smem + TC_OFF_G);  // [GD][128 threads][16]

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const int cid = static_cast<int>(ptx::cluster_id_x());
    const int direction = dir_in >= 0 ? dir_in : (cid & 1);
    const int tile = dir_in >= 0 ? cid : (cid >> 1);
    const float *__restrict__ rp = rp_in + (dir_in >= 0 ? 0 : direction * kGates * kHidden);
    const float *__restrict__ bias = bias_in + (dir_in >= 0 ? 0 : direction * kGates);
    const int tile_w0 = tile * TC_N;
    // the cells of this thread: window n of the tile, units ub .. ub + 3
    const int n = tid >> 3, quad = tid & 7;
    const int ub = 32 * static_cast<int>(rank) + 4 * quad;
    const bool valid = tile_w0 + n < batch;
    const uint32_t slice_bytes_in = 3u * TC_SLICE_BYTES;  // per step, from the 3 peers

    if (tid == 0) {
        ptx::mbar_init(&hfull[0], 1);
        ptx::mbar_init(&hfull[1], 1);
        ptx::mbar_init(mma_bar, 1);
        ptx::mbar_init(drain_bar, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        // arm buffer 1 for h_0 and buffer 0 for h_1
        if (steps > 1)
            ptx::mbar_arrive_expect_tx(&hfull[1], slice_bytes_in);
        if (steps > 2)
            ptx::mbar_arrive_expect_tx(&hfull[0], slice_bytes_in);
    }
    if (warp == 0) {
        ptx::tmem_alloc(tmem_slot, TC_TMEM_COLS);
        ptx::tmem_relinquish();
    }
    // h_{-1} = 0 in both buffers
    for (int i = tid; i < 2 * TC_B_BYTES / 16; i += TC_THREADS)
        reinterpret_cast<float4 *>(smem)[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

    // R rows into tensor memory: lane 32 q + u holds gate q of unit 32 r + u
    if constexpr (!FLOOR) {
        const int q = warp;
        const float kq = q == 2 ? K2 : K0;
        const float *src = rp + (4 * (32 * static_cast<int>(rank) + lane) + q) * kHidden;
#pragma unroll 1
        for (int cb = 0; cb < kHidden / 32; ++cb) {
            uint32_t hi[32], lo[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float v = src[32 * cb + i] * kq;
                const float h = ptx::tf32_rna(v);
                hi[i] = __float_as_uint(h);
                lo[i] = __float_as_uint(ptx::tf32_rna(v - h));
            }
            ptx::tmem_st_32x32b_x32(tmem + lane_base + TC_AHI + 32 * cb, hi);
            ptx::tmem_st_32x32b_x32(tmem + lane_base + TC_ALO + 32 * cb, lo);
        }
        ptx::tmem_st_wait();
    }
    float bias_v[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q)
            bias_v[j][q] = bias[4 * (ub + j) + q] * (q == 2 ? K2 : K0);
    // G columns of units ub .. ub + 3 (16 consecutive values) of window n
    const float *gsrc = g + direction * kGates + 4 * ub +
                        static_cast<long>(tile_w0 + n) * steps * kGateColumns;
    float *yrow = y + static_cast<long>(tile_w0 + n) * steps * kOutput + direction * kHidden + ub;

    // B buffers: [parity][slice = rank][plane][K-block of 16][16 rows x 64 B];
    // this thread's 16 bytes of h (units ub .. ub + 3, window n) in plane 0,
    // the 64-byte swizzle applied (16-byte chunk c of row n sits at
    // c ^ ((n / 2) % 4) within its 512-byte group of 8 rows)
    const uint32_t b_base = ptx::smem_u32(smem);
    const uint32_t chunk_off = rank * TC_SLICE_BYTES + (quad >> 2) * TC_KB_BYTES +
                               (n >> 3) * 512 + (n & 7) * 64 +
                               static_cast<uint32_t>(((quad & 3) ^ ((n >> 1) & 3)) * 16);

    ptx::tc_fence_before();
    // every CTA of the cluster initialised before anyone copies into it
    ptx::cluster_arrive_release();
    ptx::cluster_wait_acquire();
    ptx::tc_fence_after();
    ptx::griddep_launch_dependents();
    // launched as a programmatic dependent of the kernel that writes its
    // input: wait for that kernel's end before the first read of it
    ptx::griddep_wait();

    auto gissue = [&](int s) {
        const long t = direction ? steps - 1 - s : s;
        const bool ok = valid && s < steps;
        const float *src = ok ? gsrc + t * kGateColumns : g;
        float *dst = gring + ((s % TC_GD) * TC_THREADS + tid) * 16;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            ptx::cp_async_16(ptx::smem_u32(dst + 4 * i), ok ? src + 4 * i : g, ok ? 16u : 0u);
        ptx::cp_async_commit();
    };
    for (int s = 0; s < TC_GD; ++s)
        gissue(s);

    // bounded wait of one thread; on timeout it records the fault and the
    // abort flag, which every thread reads after the next CTA barrier
    auto wait_bounded = [&](uint64_t *bar, uint32_t parity, bool cluster_scope) -> bool {
        auto try_once = [&]() {
            return cluster_scope ? ptx::mbar_try_wait_cluster(bar, parity)
                                 : ptx::mbar_try_wait(bar, parity);
        };
        if (try_once())
            return true;
        const uint64_t start = ptx::globaltimer();
        while (!try_once()) {
            if (*abort_flag)
                return false;
            if (ptx::globaltimer() - start > wait_limit_ns) {
                atomicOr(fault, kFaultRecurrence);
                *abort_flag = 1;
                return false;
            }
        }
        return true;
    };

    float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (!(withhold && rank == 0)) {
        for (int s = 0; s < steps; ++s) {
            const int par = s & 1;
            const int t = direction ? steps - 1 - s : s;
            // 1. the peers' slices of h_{s-1} in buffer `par` (this CTA's own
            //    slice was written before the last CTA barrier); then the MMAs
            if (tid == 0) {
                bool ok = true;
                if (s > 0) {
                    ok = wait_bounded(&hfull[par], ((s - 1) >> 1) & 1, true);
                    if (ok && s + 2 < steps)
                        ptx::mbar_arrive_expect_tx(&hfull[par], slice_bytes_in);
                }
                if (ok) {
                    ptx::tc_fence_after();
                    if constexpr (!FLOOR) {
                        const uint32_t bb = b_base + static_cast<uint32_t>(par * TC_B_BYTES);
#pragma unroll
                        for (int k8 = 0; k8 < kHidden / 8; ++k8) {
                            const int kb = k8 >> 1;
                            const uint32_t bhi = bb + static_cast<uint32_t>(
                                                          (kb >> 1) * TC_SLICE_BYTES +
                                                          (kb & 1) * TC_KB_BYTES + (k8 & 1) * 32);
                            const uint32_t blo = bhi + 2 * TC_KB_BYTES;
                            ptx::mma_tf32_tmem_a(tmem + TC_D, tmem + TC_AHI + 8 * k8,
                                                 ptx::sw64_desc(bhi), TC_IDESC, k8 != 0);
                            ptx::mma_tf32_tmem_a(tmem + TC_D, tmem + TC_AHI + 8 * k8,
                                                 ptx::sw64_desc(blo), TC_IDESC, 1);
                            ptx::mma_tf32_tmem_a(tmem + TC_D, tmem + TC_ALO + 8 * k8,
                                                 ptx::sw64_desc(bhi), TC_IDESC, 1);
                        }
                    }
                    ptx::mma_commit(mma_bar);
                }
            }
            __syncthreads();
            if (*abort_flag)
                break;
            // 2. z into shared memory: warp q holds gate q of the 32 units
            //    (the tensor-memory load is warp-collective: the whole warp
            //    takes it only if every lane's wait succeeded)
            if (__all_sync(0xffffffffu, wait_bounded(mma_bar, static_cast<uint32_t>(s & 1), false))) {
                ptx::tc_fence_after();
                if constexpr (!FLOOR) {
                    uint32_t r[16];
                    ptx::tmem_ld_32x32b_x16(tmem + lane_base + TC_D, r);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < TC_N; ++j)
                        zbuf[(warp * TC_N + j) * 32 + lane] = __uint_as_float(r[j]);
                }
            }
            ptx::tc_fence_before();
            __syncthreads();
            if (*abort_flag)
                break;
            // 3. the cells of units ub .. ub + 3, window n
            ptx::cp_async_wait<TC_GD - 1>();
            const float4 *gv =
                reinterpret_cast<const float4 *>(gring + ((s % TC_GD) * TC_THREADS + tid) * 16);
            float h[4];
            if constexpr (FLOOR) {
                // the new h depends on one received value and on G only
                const float hv = *reinterpret_cast<const float *>(
                    smem + par * TC_B_BYTES + ((rank + 1) & 3) * TC_SLICE_BYTES +
                    (chunk_off - rank * TC_SLICE_BYTES));
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    h[j] = fmaf(hv, 0.5f, gv[j].x * 0.001f);
            } else {
                float4 zq[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    zq[q] = *reinterpret_cast<const float4 *>(&zbuf[(q * TC_N + n) * 32 + 4 * quad]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 gj = gv[j];  // unit ub + j, gates 0..3
                    const float zj[4] = {(&zq[0].x)[j], (&zq[1].x)[j], (&zq[2].x)[j],
                                         (&zq[3].x)[j]};
                    const float gg[4] = {gj.x, gj.y, gj.z, gj.w};
                    float a[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float w = zj[q] + fmaf(gg[q], q == 2 ? K2 : K0, bias_v[j][q]);
                        a[q] = q == 2 ? fmaf(2.0f, inv_one_plus_ex2(w), -1.0f)
                                      : inv_one_plus_ex2(w);
                    }
                    c[j] = cell_update(a[0], a[1], a[2], c[j]);
                    const float r = inv_one_plus_ex2(c[j] * (-2.0f * kLog2e));
                    h[j] = fmaf(2.0f * a[3], r, -a[3]);
                }
            }
            if (valid)
                *reinterpret_cast<float4 *>(yrow + static_cast<long>(t) * kOutput) =
                    make_float4(h[0], h[1], h[2], h[3]);
            // 4. h_s (hi, lo) into this CTA's slice of buffer par ^ 1; the
            //    slice to the peers once every thread has written it
            const bool push = s + 1 < steps;
            if (push) {
                float4 hi, lo;
                ptx::split4(make_float4(h[0], h[1], h[2], h[3]), hi, lo);
                uint8_t *dst = smem + (par ^ 1) * TC_B_BYTES + chunk_off;
                *reinterpret_cast<float4 *>(dst) = hi;
                *reinterpret_cast<float4 *>(dst + 2 * TC_KB_BYTES) = lo;
                ptx::fence_proxy_async_smem();
            }
            __syncthreads();
            if (push && tid < TC_C - 1) {
                // thread i copies the slice to the i-th other CTA
                const uint32_t peer = (rank + 1 + static_cast<uint32_t>(tid)) & (TC_C - 1);
                const uint32_t off = static_cast<uint32_t>((par ^ 1) * TC_B_BYTES) +
                                     rank * TC_SLICE_BYTES;
                ptx::bulk_copy_to_peer(ptx::map_to_rank(b_base + off, peer), b_base + off,
                                       TC_SLICE_BYTES,
                                       ptx::map_to_rank(ptx::smem_u32(&hfull[par ^ 1]), peer));
            }
            gissue(s + TC_GD);
        }
    }
    ptx::cp_async_wait_all();
    // every MMA issued has completed before tensor memory is freed
    if (tid == 0) {
        ptx::mma_commit(drain_bar);
        ptx::mbar_wait_drain(drain_bar, 0, fault, kDefaultWaitLimitNs);
    }
    ptx::tc_fence_before();
    __syncthreads();
    // no CTA leaves while a peer may still copy into its shared memory
    ptx::cluster_arrive_release();
    ptx::cluster_wait_acquire();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TC_TMEM_COLS);
    }
}

struct Variant {
    int cluster;
    int nw;       // windows per chunk
    int nch;      // chunks per lane
    int tile;     // windows per cluster
    int threads;  // per CTA
    const void *fn;
    const void *floor_fn;  // the same variant in FLOOR mode
    int smem = 0;          // dynamic shared memory per CTA
};

template <int C, int NW, int NCH = 1, int THREADS = threads_for<C>()>
Variant variant()
{
    return Variant{C, NW, NCH, THREADS / 8 / (kHidden / C) * NW * NCH, THREADS,
                   reinterpret_cast<const void *>(&recurrence_kernel<C, NW, NCH, THREADS>),
                   reinterpret_cast<const void *>(
                       &recurrence_kernel<C, NW, NCH, THREADS, true>)};
}

template <int C, int NW, int NCH>
Variant variant_u2w()
{
    return Variant{C, NW, NCH, NW * NCH, 512 / C,
                   reinterpret_cast<const void *>(&recurrence_u2w_kernel<C, NW, NCH>),
                   reinterpret_cast<const void *>(&recurrence_u2w_kernel<C, NW, NCH, true>)};
}

// "Narrow" variants (one window group per CTA: 128 threads for clusters of
// 8, 64 for clusters of 16) give each SM sub-partition fewer warps, for small
// batches where wider CTAs would mostly compute padding windows.
const Variant kVariants[] = {
    variant<16, 1>(),           variant<16, 2>(),   variant<16, 4>(),   variant<16, 8>(),
    variant<8, 1>(),            variant<8, 2>(),    variant<8, 4>(),    variant<8, 8>(),
    variant<4, 1>(),            variant<4, 2>(),    variant<2, 1>(),
    variant<4, 1, 2>(),         variant<4, 1, 4>(), variant<4, 1, 8>(), variant<4, 2, 2>(),
    variant<4, 2, 4>(),         variant<4, 2, 8>(), variant<8, 2, 4>(),
    variant<8, 1, 1, 128>(),    variant<8, 2, 1, 128>(), variant<16, 1, 1, 64>(),
    variant<16, 2, 1, 64>(),    variant<4, 4, 2>(),      variant<4, 4, 4>(),
    variant<4, 8, 1>(),         variant<4, 8, 2>(),      variant<4, 4, 1>(),
    variant<8, 4, 1, 128>(),    variant<8, 8, 1, 128>(),
    // two units per 8-lane group, one window per cluster of 64-thread CTAs
    Variant{8, 1, 1, 1, 64, reinterpret_cast<const void *>(&recurrence_u2_kernel<false>),
            reinterpret_cast<const void *>(&recurrence_u2_kernel<true>)},
    // the same in clusters of 4 CTAs of 128 threads
    Variant{4, 1, 1, 1, 128, reinterpret_cast<const void *>(&recurrence_u2_kernel<false, 4>),
            reinterpret_cast<const void *>(&recurrence_u2_kernel<true, 4>)},
    // two units per 8-lane group, several windows per lane
    variant_u2w<8, 4, 1>(), variant_u2w<8, 4, 2>(), variant_u2w<4, 4, 1>(),
    variant_u2w<4, 4, 2>(), variant_u2w<8, 8, 1>(), variant_u2w<4, 8, 1>(),
    variant_u2w<8, 8, 2>(),     variant_u2w<8, 2, 1>(), variant_u2w<8, 2, 2>(),
    variant_u2w<4, 2, 1>(),     variant_u2w<4, 2, 2>(),  variant_u2w<2, 4, 2>(),
    variant_u2w<2, 4, 1>(),
    // tensor cores: clusters of 4 CTAs of 128 threads, 16 windows per cluster
    Variant{4, 16, 1, TC_N, TC_THREADS,
            reinterpret_cast<const void *>(&recurrence_tc_kernel<false>),
            reinterpret_cast<const void *>(&recurrence_tc_kernel<true>), TC_SMEM},
};

// threads == 0: the variant's default block size
const Variant *find_variant(int cluster, int nw, int nch, int threads = 0)
{
    for (const Variant &v : kVariants)
        if (v.cluster == cluster && v.nw == nw && v.nch == nch &&
            (threads ? v.threads == threads : v.threads == (cluster == 2 ? 512 : 256)))
            return &v;
    return nullptr;
}

int max_active_clusters(const Variant &v, int *out);

// The default variant for a batch: the candidate with the least estimated
// time per step.  A launch's step time is set by how many clusters share the
// GPU: it stays flat while the clusters (both directions) fit one SM each
// way, then jumps as clusters start to share SMs (their FFMA2, shared-memory
// loads and exchanges queue behind one another).  Each candidate carries its
// measured step times (GB300, 152 SMs, both directions in one launch,
// T = 589, us) as plateaus: "up to k tiles per direction: t", including the
// second wave where a candidate stays competitive there; a batch past the
// last plateau runs as repeated waves of it.  On another SM count the tile
// counts scale with it.  Chosen this way, the step is within 1.5 % of the
// fastest candidate's at every batch from 1 to 320 windows (measured: 1-7
// windows one unit per group, 8-37 two units in clusters of 4, 38-74 two
// units and two windows per lane, 75-100 4 windows per group, 101-152 two
// units and 4 windows per lane in clusters of 2, then in clusters of 4 (two
// waves), in two chunks from 221 to 264 and in clusters of 2 from 265 to 304).
// Ties go to the earlier candidate.
const Variant *choose_variant(int batch)
{
    struct Plateau {
        int tiles;  // up to this many tiles per direction
        float us;   // time per step
    };
    struct Candidate {
        int cluster, nw, nch, threads, n;
        Plateau p[7];
    };
    static const Candidate cand[] = {
        // narrow clusters of 8, 128 threads, one window per cluster
        {8, 1, 1, 128, 6, {{4, .344f}, {7, .356f}, {11, .403f}, {18, .417f}, {25, .462f},
                           {37, .535f}}},
        // clusters of 4, 128 threads, two units per lane group (of 8 CTAs of 64
        // threads: 0.389 / 0.462 us at 8 / 32 windows against 0.365 / 0.446)
        {4, 1, 1, 128, 4, {{8, .365f}, {18, .376f}, {37, .448f}, {48, .874f}}},
        // clusters of 4, 128 threads, two units per group, 2 windows per lane
        {4, 2, 1, 128, 5, {{18, .522f}, {37, .654f}, {64, 1.253f}, {74, 1.30f}, {88, 1.87f}}},
        // clusters of 4, 128 threads, two units per group, 4 windows per lane
        {4, 4, 1, 128, 7, {{9, .716f}, {18, .748f}, {33, 1.095f}, {37, 1.179f}, {55, 1.702f},
                           {73, 2.107f}, {74, 2.29f}}},
        // narrow clusters of 8, 128 threads, 4 windows per group
        {8, 4, 1, 128, 5, {{4, .626f}, {7, .682f}, {11, .754f}, {18, .81f}, {25, 1.062f}}},
        // clusters of 4, 128 threads, two units per group, 2 chunks of 4 windows
        {4, 4, 2, 128, 3, {{18, 1.215f}, {33, 1.995f}, {37, 2.36f}}},
        // clusters of 2, 256 threads (one peer per push), two units per group,
        // 4 windows per lane, and 2 chunks of 4
        {2, 4, 1, 256, 2, {{38, 1.081f}, {76, 2.155f}}},
        {2, 4, 2, 256, 1, {{38, 2.03f}}}};
    constexpr int N = sizeof(cand) / sizeof(cand[0]);
    static std::mutex mu;
    static int fits[64][N];
    static int sms[64];
    static bool known[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return find_variant(4, 4, 1, 128);
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!known[dev]) {
            for (int i = 0; i < N; ++i) {
                int n = 0;
                const Variant *v =
                    find_variant(cand[i].cluster, cand[i].nw, cand[i].nch, cand[i].threads);
                fits[dev][i] = (v && max_active_clusters(*v, &n) == LSTM_OK) ? n : 0;
            }
            if (cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) !=
                    cudaSuccess ||
                sms[dev] <= 0)
                sms[dev] = 152;
            known[dev] = true;
        }
    }
    auto scaled = [&](int tiles) {
        return std::max(1, static_cast<int>(static_cast<long>(tiles) * sms[dev] / 152));
    };
    const Variant *best = nullptr;
    double best_cost = 0.0;
    for (int i = 0; i < N; ++i) {
        const Candidate &c = cand[i];
        const Variant *v = find_variant(c.cluster, c.nw, c.nch, c.threads);
        if (!v || fits[dev][i] < 2)
            continue;
        const long tiles = (static_cast<long>(batch) + v->tile - 1) / v->tile;
        const long last = scaled(c.p[c.n - 1].tiles);
        const long waves = (tiles + last - 1) / last;
        const long k = tiles - (waves - 1) * last;
        double cost = static_cast<double>(waves - 1) * c.p[c.n - 1].us;
        for (int j = 0; j < c.n; ++j)
            if (k <= scaled(c.p[j].tiles)) {
                cost += c.p[j].us;
                break;
            }
        if (!best || cost < best_cost) {
            best = v;
            best_cost = cost;
        }
    }
    return best ? best : find_variant(4, 4, 1, 128);
}

int launch_variant(const Variant &v, const float *g, const float *rp, const float *bias, float *y,
                   int batch, int steps, int direction, unsigned *fault, cudaStream_t stream,
                   bool floor = false, bool pdl = false)
{
    const long tiles = (static_cast<long>(batch) + v.tile - 1) / v.tile;
    const long blocks = tiles * v.cluster * (direction == kBothDirections ? 2 : 1);
    if (blocks > 0x7fffffffL)
        return fail(LSTM_E_OVERFLOW, "recurrence: %d windows need %ld blocks", batch, blocks);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(static_cast<unsigned>(v.threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(v.smem);
    cfg.stream = stream;
    // Normally launched after the kernel before it has ended: started early
    // (programmatic dependent launch) while that kernel covers the GPU, the
    // clusters were placed on the SMs it had already left, several to an SM,
    // and the whole layer ran at the pace of the most crowded SM (b32_t589:
    // 2.23 instead of 1.36 ms per forward).  `pdl` (both grids fit side by
    // side): started early, so the set-up overlaps that kernel.
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(v.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    // failure-test settings (kernel parameters: reading them from a device
    // variable at kernel start measured 3-7 % slower per step)
    KernelTest test = kernel_test(kTestRecurrence);
    int st;
    if ((st = check_launch_injection("recurrence launch")))
        return st;
    void *args[] = {const_cast<float **>(&g), const_cast<float **>(&rp),
                    const_cast<float **>(&bias), &y, &batch, &steps, &direction, &fault,
                    &test.wait_limit_ns, &test.withhold};
    return cuda_status(cudaLaunchKernelExC(&cfg, floor ? v.floor_fn : v.fn, args),
                       "recurrence launch");
}

} // namespace

int recurrence_prepare(int)
{
    for (const Variant &v : kVariants) {
        if (v.smem > 48 * 1024) {
            for (const void *fn : {v.fn, v.floor_fn}) {
                int st = cuda_status(cudaFuncSetAttribute(fn,
                                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                          v.smem),
                                     "recurrence shared-memory attribute");
                if (st != LSTM_OK)
                    return st;
            }
        }
        if (v.cluster > 8) {
            for (const void *fn : {v.fn, v.floor_fn}) {
                int st = cuda_status(
                    cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
                    "recurrence cluster-size attribute");
                if (st != LSTM_OK)
                    return st;
            }
        }
    }
    return LSTM_OK;
}

int launch_recurrence(const float *g, const float *rp, const float *bias, float *y, int batch,
                      int steps, int direction, unsigned *fault, cudaStream_t stream,
                      int co_resident_ctas)
{
    const Variant &v = *choose_variant(batch);
    bool pdl = false;
    if (co_resident_ctas >= 0) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) {
            const long tiles = (static_cast<long>(batch) + v.tile - 1) / v.tile;
            const long blocks = tiles * v.cluster * (direction == kBothDirections ? 2 : 1);
            pdl = blocks + co_resident_ctas <= sms;
        }
    }
    return launch_variant(v, g, rp, bias, y, batch, steps, direction, fault, stream, false, pdl);
}

int launch_recurrence_floor(const float *g, const float *rp, const float *bias, float *y,
                            int batch, int steps, int direction, unsigned *fault,
                            cudaStream_t stream)
{
    return launch_variant(*choose_variant(batch), g, rp, bias, y, batch, steps, direction, fault,
                          stream, true);
}

int recurrence_fused_max_clusters(int kp, int *out)
{
    const void *fn = kp <= 64 ? reinterpret_cast<const void *>(&recurrence_fused_kernel<64>)
                              : reinterpret_cast<const void *>(&recurrence_fused_kernel<256>);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(8);
    cfg.blockDim = dim3(256);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 8;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaOccupancyMaxActiveClusters(out, fn, &cfg), "fused max active clusters");
}

int launch_recurrence_fused(const float *x, int in_width, const float *wp_hi, const float *wp_lo,
                            int kp, const float *rp, const float *bias, float *y, int batch,
                            int steps, int direction, unsigned *fault, cudaStream_t stream)
{
    if (kp != 64 && kp != 256)
        return fail(LSTM_E_INVALID, "fused recurrence: kp %d (64 or 256)", kp);
    if (in_width <= 0 || in_width > kp || in_width % 4 != 0)
        return fail(LSTM_E_INVALID, "fused recurrence: in_width %d (a multiple of 4 up to kp %d)",
                    in_width, kp);
    const long blocks = static_cast<long>(batch) * 8 * (direction == kBothDirections ? 2 : 1);
    if (blocks > 0x7fffffffL)
        return fail(LSTM_E_OVERFLOW, "fused recurrence: %d windows", batch);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 8;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    KernelTest test = kernel_test(kTestRecurrence);
    int st;
    if ((st = check_launch_injection("fused recurrence launch")))
        return st;
    void *args[] = {const_cast<float **>(&x), &in_width, const_cast<float **>(&wp_hi),
                    const_cast<float **>(&wp_lo), const_cast<float **>(&rp),
                    const_cast<float **>(&bias), &y, &batch, &steps, &direction, &fault,
                    &test.wait_limit_ns, &test.withhold};
    const void *fn = kp == 64 ? reinterpret_cast<const void *>(&recurrence_fused_kernel<64>)
                              : reinterpret_cast<const void *>(&recurrence_fused_kernel<256>);
    return cuda_status(cudaLaunchKernelExC(&cfg, fn, args), "fused recurrence launch");
}

int launch_recurrence_variant(const float *g, const float *rp, const float *bias, float *y,
                              int batch, int steps, int direction, int cluster, int nw, int nch,
                              int threads, unsigned *fault, cudaStream_t stream)
{
    const Variant *v = find_variant(cluster, nw, nch, threads);
    if (!v)
        return fail(LSTM_E_INVALID,
                    "recurrence: no variant with cluster %d, %d windows per chunk, %d chunks, "
                    "%d threads",
                    cluster, nw, nch, threads);
    return launch_variant(*v, g, rp, bias, y, batch, steps, direction, fault, stream);
}

int recurrence_max_clusters(int cluster, int nw, int nch, int threads, int *out)
{
    const Variant *v = find_variant(cluster, nw, nch, threads);
    if (!v)
        return fail(LSTM_E_INVALID,
                    "recurrence: no variant with cluster %d, %d windows per chunk, %d chunks, "
                    "%d threads",
                    cluster, nw, nch, threads);
    return max_active_clusters(*v, out);
}

namespace {
int max_active_clusters(const Variant &vr, int *out)
{
    const Variant *v = &vr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(v->cluster));
    cfg.blockDim = dim3(static_cast<unsigned>(v->threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(v->smem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(v->cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaOccupancyMaxActiveClusters(out, v->fn, &cfg), "max active clusters");
}
}  // namespace

} // namespace lstm
