// Router: logits = x . W_g (fp32 accumulation), top-k selection (ties to the
// lower expert index) and the gates ("Mixtral of Experts" (azimuth.plus),
// router paragraph).
//
// One block handles TB tokens (2, 4 or 8).  Its 256 threads split the hidden
// dimension: thread i takes 16-byte slices i, i + 256, ... of every token row
// and the same slices of each expert's router row, issues a pass's loads
// before any arithmetic, and the block reduces the per-thread partial sums in
// a fixed order (butterfly in each warp, then warps in order).  HBM traffic is
// x once; the router matrix is served from L1/L2 and unpacked once per TB
// tokens.
//
// Fused RMSNorm (pre-norm blocks): a first pass over the rows gives each
// token's RMSNorm scale (stored for the grouping pass); the logits are then
// taken of round(x * scale), the normalised row the stand-alone RMSNorm
// kernel would have stored, read again from L1.
//
// Large bf16 batches (from four tokens per SM, up to 8 experts) go to
// router_wide_kernel, which streams the token rows through shared memory with
// bulk copies and keeps the router rows in registers; it sums in the same
// order, so the logits are the same bits either way.
#include <stdio.h>
#include <stdlib.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kRouterThreads = kNormThreads;

// Selection and gates for one token, written out (KMAX >= k slots).
template <int KMAX>
__device__ __forceinline__ void select_and_store(const float *l, int t, int E, int k, int gating,
                                                 int *idx, float *gates) {
    int sel[KMAX];
    float g[KMAX];
    topk_gates<KMAX>(l, E, k, gating, sel, g);
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        if (j < k) {
            idx[(size_t)t * k + j] = sel[j];
            gates[(size_t)t * k + j] = g[j];
        }
    }
}

// Bias, selection, gates and outputs for one token, from its E logits.
__device__ __forceinline__ void finish_token(float *l, const float *bias, int t, int E, int k,
                                             int gating, float *logits, int *idx, float *gates) {
    for (int e = 0; e < E; ++e) {
        l[e] += (bias != nullptr ? bias[e] : 0.f);
        logits[(size_t)t * E + e] = l[e];
    }
    if (k <= 2)
        select_and_store<2>(l, t, E, k, gating, idx, gates);
    else
        select_and_store<MOE_MAX_TOPK>(l, t, E, k, gating, idx, gates);
}

// Experts are taken EG at a time (one pass over the token rows per group,
// the later passes hitting L1).  V: 16-byte slices per thread per pass, all
// of a pass's loads in flight together.  Rows of experts >= E are clamped to
// a valid row and their sums ignored, which keeps the loads free of branches.
// NORM: the fused RMSNorm (eps; each token's scale written to inv_rms).
// x_copy != nullptr (one pass over the rows: EG >= E): x is page-locked host
// memory read over the bus, and each block also writes its rows to x_copy
// in device memory for the kernels after it.
template <typename T, int TB, int EG, int V, bool NORM>
__global__ void __launch_bounds__(kRouterThreads) router_kernel(
    const T *__restrict__ x, const T *__restrict__ Wg, const float *__restrict__ bias, int Tn,
    int d, int E, int k, int gating, float eps, float *inv_rms, float *logits, int *idx,
    float *gates, T *x_copy) {
    constexpr int VN = Vec<T>::n;
    constexpr int NW = kRouterThreads / 32;
    __shared__ float s_part[NW][TB][MOE_MAX_EXPERTS];
    __shared__ float s_l[TB][MOE_MAX_EXPERTS];
    __shared__ float s_ss[NW][TB];
    __shared__ float s_scale[TB];

    pdl_wait();
    pdl_trigger();
    const int t0 = blockIdx.x * TB;
    const int nt = min(TB, Tn - t0);
    const int nvec = d / VN;
    const uint4 *xr[TB];
#pragma unroll
    for (int j = 0; j < TB; ++j)  // rows past the batch repeat its last token (results unused)
        xr[j] = reinterpret_cast<const uint4 *>(x + (size_t)(t0 + min(j, nt - 1)) * d);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    float sc[TB];
#pragma unroll
    for (int j = 0; j < TB; ++j) sc[j] = 1.f;
    if (NORM) {
        float ss[TB];
#pragma unroll
        for (int j = 0; j < TB; ++j) ss[j] = 0.f;
        for (int v = threadIdx.x; v < nvec; v += kRouterThreads) {
#pragma unroll
            for (int j = 0; j < TB; ++j) ss[j] = slice_sumsq<T>(ss[j], xr[j][v]);
        }
        {
            constexpr int kShiftT = TB == 8 ? 2 : TB == 4 ? 3 : TB == 2 ? 4 : 5;
            const float tot = warp_reduce_scatter<TB>(ss, lane);
            if ((lane & ((1 << kShiftT) - 1)) == 0) s_ss[warp][lane >> kShiftT] = tot;
        }
        __syncthreads();
        if (threadIdx.x < TB) {
            float tot = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < NW; ++w2) tot += s_ss[w2][threadIdx.x];
            const float scale = rms_scale(tot, d, eps);
            s_scale[threadIdx.x] = scale;
            if ((int)threadIdx.x < nt) inv_rms[t0 + threadIdx.x] = scale;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < TB; ++j) sc[j] = s_scale[j];
    }

    for (int g0 = 0; g0 < E; g0 += EG) {
        const uint4 *wr[EG];
#pragma unroll
        for (int e = 0; e < EG; ++e)
            wr[e] = reinterpret_cast<const uint4 *>(Wg + (size_t)(g0 + e < E ? g0 + e : E - 1) * d);
        float acc[TB][EG];
#pragma unroll
        for (int j = 0; j < TB; ++j)
#pragma unroll
            for (int e = 0; e < EG; ++e) acc[j][e] = 0.f;
        for (int v0 = threadIdx.x; v0 < nvec; v0 += kRouterThreads * V) {
            uint4 xs[V][TB], w[V][EG];
#pragma unroll
            for (int u = 0; u < V; ++u) {
                const int v = v0 + kRouterThreads * u;
                const int vv = v < nvec ? v : 0;
                // one pass over the rows streams them; with several passes
                // (experts taken EG at a time) they are kept for the next pass
#pragma unroll
                for (int j = 0; j < TB; ++j)
                    xs[u][j] = v < nvec ? (x_copy != nullptr ? xr[j][vv]
                                           : EG >= E ? __ldcs(xr[j] + vv) : __ldg(xr[j] + vv))
                                        : zero;
                if (x_copy != nullptr && v < nvec) {
#pragma unroll
                    for (int j = 0; j < TB; ++j)
                        if (j < nt)
                            reinterpret_cast<uint4 *>(x_copy + (size_t)(t0 + j) * d)[v] = xs[u][j];
                }
#pragma unroll
                for (int e = 0; e < EG; ++e) w[u][e] = __ldg(wr[e] + vv);
            }
#pragma unroll
            for (int u = 0; u < V; ++u) {
                float a[TB][VN];
#pragma unroll
                for (int j = 0; j < TB; ++j)
                    Vec<T>::unpack(NORM ? scale_slice<T>(xs[u][j], sc[j]) : xs[u][j], a[j]);
#pragma unroll
                for (int e = 0; e < EG; ++e) {
                    float wf[VN];
                    Vec<T>::unpack(w[u][e], wf);
#pragma unroll
                    for (int i = 0; i < VN; ++i)
#pragma unroll
                        for (int j = 0; j < TB; ++j) acc[j][e] = fmaf(a[j][i], wf[i], acc[j][e]);
                }
            }
        }
        // the warp's sums (the butterfly's bits), one (token, expert) per lane
        // or lane pair; those lanes park them
        constexpr int NV = TB * EG;
        static_assert(NV <= 32 && (NV & (NV - 1)) == 0, "token x expert sums per warp");
        float flat[NV];
#pragma unroll
        for (int j = 0; j < TB; ++j)
#pragma unroll
            for (int e = 0; e < EG; ++e) flat[j * EG + e] = acc[j][e];
        const float sum = warp_reduce_scatter<NV>(flat, lane);
        constexpr int kShift = NV == 32 ? 0 : NV == 16 ? 1 : NV == 8 ? 2 : NV == 4 ? 3 : NV == 2 ? 4 : 5;
        if ((lane & ((1 << kShift) - 1)) == 0) {
            const int o = lane >> kShift;
            const int j = o / EG, e = o - (o / EG) * EG;
            if (g0 + e < E) s_part[warp][j][g0 + e] = sum;
        }
    }
    __syncthreads();
    // warps added in order: one thread per (token, expert)
    for (int i = threadIdx.x; i < TB * E; i += kRouterThreads) {
        const int j = i / E, e = i - j * E;
        float s = s_part[0][j][e];
#pragma unroll
        for (int w2 = 1; w2 < NW; ++w2) s += s_part[w2][j][e];
        s_l[j][e] = s;
    }
    __syncthreads();
    if ((int)threadIdx.x < nt)
        finish_token(s_l[threadIdx.x], bias, t0 + threadIdx.x, E, k, gating, logits, idx, gates);
}

// Router for large batches (bf16, E <= 8, d <= 2 * 256 slices of 8): a
// persistent grid of one block per SM, warp-specialised around mbarriers.
//   warps 0..7  compute: the logits' partial sums of a group of kWideTB
//               consecutive tokens, from shared memory; each thread keeps its
//               slices of the router matrix in registers for the whole run
//   warp 8      lane 0 issues the bulk copies (cp.async.bulk), each group's
//               rows (one contiguous chunk of x) into a ring of kWideStages
//               stages, as soon as a stage is free
//   warp 9      adds the compute warps' sums and writes each token's logits,
//               choices and gates, from a ring of kWideSums sum buffers
// The compute warps meet at no block barrier (with NORM, once a group over
// the row sums of squares), so the selection and the stores of one group
// overlap the products of the next, and up to kWideStages - 1 groups of rows
// are in flight per SM.  Compute thread i takes the same slices i, i + 256 of
// every row as router_kernel and sums in the same order (slices, then
// elements, in order; the butterfly's sums via warp_reduce_scatter; warps in
// order), so the logits -- and, with NORM, the RMSNorm scales -- are the same
// bits as router_kernel's.  The products are issued two experts at a time as
// packed fp32x2 FMAs, each lane of which rounds exactly as a scalar fmaf.
constexpr int kWideTB = 4;
constexpr int kWideE = 8;
constexpr int kWideNS = 2;      // slices per thread and row (d <= 4096 in bf16)
constexpr int kWideStages = 6;  // ring stages of kWideTB rows
constexpr int kWideSums = 4;    // sum buffers between the compute warps and warp 9
constexpr int kWideCompute = kRouterThreads;
constexpr int kWideThreads = kWideCompute + 64;

// dynamic shared memory: the ring
__host__ __device__ constexpr size_t wide_smem_bytes(int d) {
    return (size_t)kWideStages * kWideTB * d * 2;
}

// Element h (0: low half, 1: high half) of a word of two bf16 values, as
// Vec<bf16>::unpack gives it.
__device__ __forceinline__ float bf16_word_elt(uint32_t w, int h) {
    return __uint_as_float(h ? (w & 0xFFFF0000u) : (w << 16));
}

// bar.red.and over the compute warps (named barrier 1): every compute thread
// gets the AND of all their flags
__device__ __forceinline__ bool compute_warps_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kWideCompute)
        : "memory");
    return r != 0;
}

template <bool NORM>
__global__ void __launch_bounds__(kWideThreads, 1) router_wide_kernel(
    const __nv_bfloat16 *__restrict__ x, const __nv_bfloat16 *__restrict__ Wg,
    const float *__restrict__ bias, int Tn, int d, int E, int k, int gating, float eps,
    float *inv_rms, float *logits, int *idx, float *gates, int *status,
    unsigned long long wait_limit_ns) {
    constexpr int NW = kWideCompute / 32;
    constexpr int EP = kWideE / 2;  // expert pairs
    extern __shared__ __align__(128) uint4 s_ring[];  // [kWideStages][kWideTB][nvec]
    __shared__ float s_part[kWideSums][NW][kWideTB][kWideE];
    __shared__ float s_ss[2][NW][kWideTB];
    __shared__ __align__(8) uint64_t s_full[kWideStages], s_empty[kWideStages];
    __shared__ __align__(8) uint64_t s_sfull[kWideSums], s_sempty[kWideSums];
    __shared__ int s_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nvec = d / 8;
    const int ngroups = (Tn + kWideTB - 1) / kWideTB;
    const int nlocal = blockIdx.x < ngroups ? (ngroups - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    volatile int *abort = &s_abort;

    if (threadIdx.x == 0) {
        // the compute warps arrive once per warp (lane 0, after __syncwarp)
        for (int st = 0; st < kWideStages; ++st) {
            ptx::mbar_init(&s_full[st], 1);
            ptx::mbar_init(&s_empty[st], NW);
        }
        for (int b = 0; b < kWideSums; ++b) {
            ptx::mbar_init(&s_sfull[b], NW);
            ptx::mbar_init(&s_sempty[b], 1);
        }
        s_abort = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();

    if (warp == NW) {
        // ---- bulk copies: local group i is group blockIdx.x + i * gridDim.x,
        //      in stage i % kWideStages ----
        if (lane != 0) return;
        auto issue = [&](int i) {
            const int t0 = (blockIdx.x + i * gridDim.x) * kWideTB;
            const uint32_t bytes = (uint32_t)min(kWideTB, Tn - t0) * (uint32_t)d * 2u;
            uint64_t *bar = &s_full[i % kWideStages];
            ptx::mbar_arrive_expect_tx(bar, bytes);
            ptx::bulk_load_1d(s_ring + (size_t)(i % kWideStages) * kWideTB * nvec,
                              x + (size_t)t0 * d, bytes, bar);
        };
        int issued = 0;
        for (; issued < kWideStages && issued < nlocal; ++issued) issue(issued);
        for (; issued < nlocal; ++issued) {
            // stage of group issued - stages: free once the compute warps are done with it
            const int j = issued - kWideStages;
            if (!ptx::mbar_wait_bounded(&s_empty[j % kWideStages], (uint32_t)(j / kWideStages) & 1u,
                                        abort, status, kStatusProducerWait, wait_limit_ns))
                break;
            issue(issued);
        }
        if (*abort) {
            // a wait expired somewhere: let the copies still in flight land
            // before the block's shared memory is released
            for (int j = issued - kWideStages; j < issued; ++j)
                if (j >= 0 && !ptx::mbar_wait_bounded(&s_full[j % kWideStages],
                                                      (uint32_t)(j / kWideStages) & 1u, nullptr,
                                                      status, kStatusDrainWait, wait_limit_ns))
                    break;
        }
        return;
    }
    if (warp == NW + 1) {
        // ---- the tokens' sums, selections and gates ----
        static_assert(kWideTB * kWideE == 32, "one lane per (token, expert) of a group");
        const int fj = lane >> 3, fe = lane & 7;
        // the bias term of finish_token (0 without a bias)
        const float bias_e = bias != nullptr && fe < E ? bias[fe] : 0.f;
        for (int i = 0; i < nlocal; ++i) {
            const int b = i % kWideSums;
            if (!__all_sync(0xffffffffu, ptx::mbar_wait_bounded(
                                             &s_sfull[b], (uint32_t)(i / kWideSums) & 1u, abort,
                                             status, kStatusEpilogueWait, wait_limit_ns)))
                break;
            const int t0 = (blockIdx.x + i * gridDim.x) * kWideTB;
            const int nt = min(kWideTB, Tn - t0);
            // one lane per (token j, expert e): the warps' sums added in
            // order, the bias, the logit written out
            float t = s_part[b][0][fj][fe];
#pragma unroll
            for (int w2 = 1; w2 < NW; ++w2) t += s_part[b][w2][fj][fe];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&s_sempty[b]);
            const float l = t + bias_e;
            if (fj < nt && fe < E) logits[(size_t)(t0 + fj) * E + fe] = l;
            // the token's logits gathered in registers by its lane e = 0,
            // which selects and writes the choices and gates
            float lv[kWideE];
#pragma unroll
            for (int e2 = 0; e2 < kWideE; ++e2)
                lv[e2] = __shfl_sync(0xffffffffu, l, (lane & ~7) | e2);
            if (fe == 0 && fj < nt) {
                const size_t o = (size_t)(t0 + fj) * k;
                if (k <= 2) {
                    int sel[2];
                    float g[2];
                    topk_gates_from<2, kWideE>([&](int e2) { return lv[e2]; }, E, k, gating, sel,
                                               g);
#pragma unroll
                    for (int q = 0; q < 2; ++q)
                        if (q < k) {
                            idx[o + q] = sel[q];
                            gates[o + q] = g[q];
                        }
                } else {
                    int sel[MOE_MAX_TOPK];
                    float g[MOE_MAX_TOPK];
                    topk_gates_from<MOE_MAX_TOPK, kWideE>([&](int e2) { return lv[e2]; }, E, k,
                                                          gating, sel, g);
#pragma unroll
                    for (int q = 0; q < MOE_MAX_TOPK; ++q)
                        if (q < k) {
                            idx[o + q] = sel[q];
                            gates[o + q] = g[q];
                        }
                }
            }
        }
        return;
    }

    // ---- compute warps ----
    // this thread's slices of the router rows (rows past E read as zero)
    uint4 wr[kWideNS][kWideE];
#pragma unroll
    for (int sl = 0; sl < kWideNS; ++sl) {
        const int v = threadIdx.x + kWideCompute * sl;
#pragma unroll
        for (int e = 0; e < kWideE; ++e)
            wr[sl][e] = v < nvec && e < E ? __ldg(reinterpret_cast<const uint4 *>(Wg) +
                                                  (size_t)e * nvec + v)
                                          : make_uint4(0, 0, 0, 0);
    }
    bool ok = true;
    for (int i = 0; i < nlocal; ++i) {
        const int st = i % kWideStages, b = i % kWideSums;
        const int t0 = (blockIdx.x + i * gridDim.x) * kWideTB;
        const int nt = min(kWideTB, Tn - t0);
        ok = ok && ptx::mbar_wait_bounded(&s_full[st], (uint32_t)(i / kWideStages) & 1u, abort,
                                          status, kStatusMmaWait, wait_limit_ns);
        // sum buffer b is free once warp 9 has read group i - kWideSums
        if (i >= kWideSums)
            ok = ok && ptx::mbar_wait_bounded(&s_sempty[b], ((uint32_t)(i / kWideSums) & 1u) ^ 1u,
                                              abort, status, kStatusMmaWait, wait_limit_ns);
        // a warp leaves the loop as a whole (its lanes meet at __syncwarp below)
        ok = __all_sync(0xffffffffu, ok);
        const uint4 *xs = s_ring + (size_t)st * kWideTB * nvec;
        float sc[kWideTB];
#pragma unroll
        for (int j = 0; j < kWideTB; ++j) sc[j] = 1.f;
        if (NORM) {
            float ss[kWideTB];
#pragma unroll
            for (int j = 0; j < kWideTB; ++j) {
                ss[j] = 0.f;
#pragma unroll
                for (int sl = 0; sl < kWideNS; ++sl) {
                    const int v = threadIdx.x + kWideCompute * sl;
                    if (v < nvec) ss[j] = slice_sumsq<__nv_bfloat16>(ss[j], xs[j * nvec + v]);
                }
            }
            const float tot = warp_reduce_scatter<kWideTB>(ss, lane);
            if ((lane & 7) == 0) s_ss[i & 1][warp][lane >> 3] = tot;
            // every compute warp leaves together when a wait failed
            if (!compute_warps_and(ok)) {
                *abort = 1;
                break;
            }
#pragma unroll
            for (int j = 0; j < kWideTB; ++j) {
                float t = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < NW; ++w2) t += s_ss[i & 1][w2][j];
                sc[j] = rms_scale(t, d, eps);
            }
#pragma unroll
            for (int j = 0; j < kWideTB; ++j)
                if ((int)threadIdx.x == j && j < nt) inv_rms[t0 + j] = sc[j];
        } else if (!ok) {
            break;
        }
        float2 acc[kWideTB][EP];
#pragma unroll
        for (int j = 0; j < kWideTB; ++j)
#pragma unroll
            for (int p = 0; p < EP; ++p) acc[j][p] = make_float2(0.f, 0.f);
#pragma unroll
        for (int sl = 0; sl < kWideNS; ++sl) {
            const int v = threadIdx.x + kWideCompute * sl;
            if (v >= nvec) break;
            uint32_t xw[kWideTB][4];  // the slice of each row, bf16 pairs
#pragma unroll
            for (int j = 0; j < kWideTB; ++j) {
                const uint4 q = NORM ? scale_slice<__nv_bfloat16>(xs[j * nvec + v], sc[j])
                                     : xs[j * nvec + v];
                xw[j][0] = q.x;
                xw[j][1] = q.y;
                xw[j][2] = q.z;
                xw[j][3] = q.w;
            }
            // element by element (the order of every sum): x of the four
            // rows, then the expert pairs
#pragma unroll
            for (int e8 = 0; e8 < 8; ++e8) {
                const int wd = e8 >> 1;
                float2 a2[kWideTB];
#pragma unroll
                for (int j = 0; j < kWideTB; ++j) {
                    const float a = bf16_word_elt(xw[j][wd], e8 & 1);
                    a2[j] = make_float2(a, a);
                }
#pragma unroll
                for (int p = 0; p < EP; ++p) {
                    const uint4 &q0 = wr[sl][2 * p], &q1 = wr[sl][2 * p + 1];
                    const uint32_t u0 = wd == 0 ? q0.x : wd == 1 ? q0.y : wd == 2 ? q0.z : q0.w;
                    const uint32_t u1 = wd == 0 ? q1.x : wd == 1 ? q1.y : wd == 2 ? q1.z : q1.w;
                    const float2 w2 =
                        make_float2(bf16_word_elt(u0, e8 & 1), bf16_word_elt(u1, e8 & 1));
#pragma unroll
                    for (int j = 0; j < kWideTB; ++j) acc[j][p] = __ffma2_rn(a2[j], w2, acc[j][p]);
                }
            }
        }
        // the warp is done with stage st (every lane's reads have returned:
        // their values fed the FMAs above)
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&s_empty[st]);
        float flat[kWideTB * kWideE];
#pragma unroll
        for (int j = 0; j < kWideTB; ++j)
#pragma unroll
            for (int p = 0; p < EP; ++p) {
                flat[j * kWideE + 2 * p] = acc[j][p].x;
                flat[j * kWideE + 2 * p + 1] = acc[j][p].y;
            }
        const float sum = warp_reduce_scatter<kWideTB * kWideE>(flat, lane);
        s_part[b][warp][lane >> 3][lane & 7] = sum;
        // the warp's sums are in place: __syncwarp orders every lane's store
        // before lane 0's (releasing) arrival
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&s_sfull[b]);
    }
}

// Selection from given logits: one thread per token.
__global__ void __launch_bounds__(128) topk_kernel(const float *__restrict__ logits, int Tn, int E,
                                                   int k, int gating, int *idx, float *gates) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x * 128 + threadIdx.x;
    if (t >= Tn) return;
    const float *l = logits + (size_t)t * E;
    if (k <= 2)
        select_and_store<2>(l, t, E, k, gating, idx, gates);
    else
        select_and_store<MOE_MAX_TOPK>(l, t, E, k, gating, idx, gates);
}

template <typename T, int TB, int EG, int V, bool NORM>
cudaError_t router_launch(const void *x, const void *Wg, const float *bias, int T_, int d, int E,
                          int k, int gating, float eps, float *inv_rms, float *logits, int *idx,
                          float *gates, cudaStream_t s, void *x_copy) {
    if (x_copy != nullptr && (EG < E || NORM)) return cudaErrorInvalidValue;
    const int grid = (T_ + TB - 1) / TB;
    return launch_pdl(router_kernel<T, TB, EG, V, NORM>, grid, kRouterThreads, 0, s,
                      static_cast<const T *>(x), static_cast<const T *>(Wg), bias, T_, d, E, k,
                      gating, eps, inv_rms, logits, idx, gates, static_cast<T *>(x_copy));
}

// Tokens per block: 2 for small batches (blocks for every SM), 4 or 8 once
// there are at least two blocks per SM, so a block reads and unpacks the
// router matrix once for more tokens.  16-byte loads in flight per thread per
// pass: V * (TB + EG).  Every choice sums each token's products in the same
// order, so a token's logits do not depend on the batch it comes in.
template <typename T, bool NORM>
cudaError_t router_dispatch_n(const void *x, const void *Wg, const float *bias, int T_, int d,
                              int E, int k, int gating, float eps, float *inv_rms, float *logits,
                              int *idx, float *gates, cudaStream_t s, void *x_copy) {
#define MOE_ROUTER(TB, EG, V)                                                                      \
    return router_launch<T, TB, EG, V, NORM>(x, Wg, bias, T_, d, E, k, gating, eps, inv_rms,      \
                                             logits, idx, gates, s, x_copy)
    // MOE_ROUTER_CFG=TB,EG,V picks one of the configurations below (measurement only)
    if (const char *c = x_copy == nullptr ? getenv("MOE_ROUTER_CFG") : nullptr) {
        int tb = 0, eg = 0, v = 0;
        if (sscanf(c, "%d,%d,%d", &tb, &eg, &v) == 3) {
            if (tb == 2 && eg == 8 && v == 2) MOE_ROUTER(2, 8, 2);
            if (tb == 2 && eg == 8 && v == 4) MOE_ROUTER(2, 8, 4);
            if (tb == 4 && eg == 8 && v == 1) MOE_ROUTER(4, 8, 1);
            if (tb == 4 && eg == 8 && v == 2) MOE_ROUTER(4, 8, 2);
            if (tb == 8 && eg == 4 && v == 1) MOE_ROUTER(8, 4, 1);
            if (tb == 8 && eg == 4 && v == 2) MOE_ROUTER(8, 4, 2);
            if (tb == 4 && eg == 4 && v == 2) MOE_ROUTER(4, 4, 2);
            if (tb == 8 && eg == 2 && v == 2) MOE_ROUTER(8, 2, 2);
            if (tb == 16 && eg == 2 && v == 1) MOE_ROUTER(16, 2, 1);
        }
    }
    // Measured (B300, d = 4096, 8 experts, CUDA graph of 50 calls): T=16 (2,8,2)
    // 3.2 us; T=1024 (2,8,2) 7.7, (4,8,1) 6.2, (8,4,1) 6.4; T=2048 (4,8,1) 10.2,
    // (8,4,1) 8.8; T=4096 (4,8,1) 17.3, (8,4,1) 15.9; T=16384 (4,8,1) 66.0,
    // (8,4,1) 57.2 us.  (From 592 tokens the streaming router_wide_kernel
    // takes bf16 batches of up to 8 experts.)
    const int blocks_per_sm = 2;
    if (E <= 8) {
        if (T_ >= 1536) MOE_ROUTER(8, 4, 1);
        if (T_ >= 4 * kPlanSms) MOE_ROUTER(4, 8, 1);
        MOE_ROUTER(2, 8, 2);
    }
    if (T_ >= 4 * blocks_per_sm * kPlanSms) MOE_ROUTER(4, 8, 1);
    MOE_ROUTER(2, 16, 1);
#undef MOE_ROUTER
}

// The streaming large-batch router where it applies (bf16, E <= 8, d <= 4096,
// from one group of four tokens per SM); MOE_ROUTER_WIDE=0|1 forces it off or
// on where it applies (measurement only).  Measured (B300, d = 4096, 8
// experts, CUDA graph of 50 calls, x resident in L2; router_kernel's best
// configuration against this one): T=592 6.4 / 4.7 us, T=1024 6.7 / 6.0,
// T=2048 9.4 / 8.6, T=4096 17.7 / 12.9, T=8192 30.4 / 22.0, T=16384 63.3 /
// 43.8 us.
constexpr int kWideMinTokens = 4 * kPlanSms;

template <bool NORM>
bool router_wide(const void *x, const void *Wg, const float *bias, int T_, int d, int E, int k,
                 int gating, float eps, float *inv_rms, float *logits, int *idx, float *gates,
                 cudaStream_t s, cudaError_t *err) {
    if (E > kWideE || d % 8 != 0 || d / 8 > kWideNS * kRouterThreads) return false;
    const int ngroups = (T_ + kWideTB - 1) / kWideTB;
    bool on = T_ >= kWideMinTokens;
    if (const char *v = getenv("MOE_ROUTER_WIDE")) on = atoi(v) != 0;
    if (!on) return false;
    const int sms = device_sm_count();
    const int grid = ngroups < sms ? ngroups : sms;
    int *status = device_status_ptr();
    if (status == nullptr) {
        *err = cudaErrorInvalidValue;
        return true;
    }
    static bool attr_done[2][64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *err = cudaErrorInvalidDevice;
        return true;
    }
    if (!attr_done[NORM][dev]) {
        if ((*err = cudaFuncSetAttribute(
                 router_wide_kernel<NORM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                 static_cast<int>(wide_smem_bytes(kWideNS * kRouterThreads * 8)))) != cudaSuccess)
            return true;
        attr_done[NORM][dev] = true;
    }
    *err = launch_pdl(router_wide_kernel<NORM>, grid, kWideThreads, wide_smem_bytes(d), s,
                      static_cast<const __nv_bfloat16 *>(x),
                      static_cast<const __nv_bfloat16 *>(Wg), bias, T_, d, E, k, gating, eps,
                      inv_rms, logits, idx, gates, status, kWaitLimitNs);
    return true;
}

template <typename T>
cudaError_t router_dispatch(const void *x, const void *Wg, const float *bias, int T_, int d,
                            int E, int k, int gating, float eps, float *inv_rms, float *logits,
                            int *idx, float *gates, cudaStream_t s, void *x_copy) {
    if (x_copy != nullptr) {
        // host rows: the single-pass configurations only
        if (E > 8 || T_ >= 1536 || inv_rms != nullptr) return cudaErrorInvalidValue;
        return router_dispatch_n<T, false>(x, Wg, bias, T_, d, E, k, gating, eps, inv_rms,
                                           logits, idx, gates, s, x_copy);
    }
    if (sizeof(T) == 2) {
        cudaError_t err = cudaSuccess;
        const bool done =
            inv_rms != nullptr
                ? router_wide<true>(x, Wg, bias, T_, d, E, k, gating, eps, inv_rms, logits, idx,
                                    gates, s, &err)
                : router_wide<false>(x, Wg, bias, T_, d, E, k, gating, eps, inv_rms, logits, idx,
                                     gates, s, &err);
        if (done) return err;
    }
    if (inv_rms != nullptr)
        return router_dispatch_n<T, true>(x, Wg, bias, T_, d, E, k, gating, eps, inv_rms, logits,
                                          idx, gates, s, nullptr);
    return router_dispatch_n<T, false>(x, Wg, bias, T_, d, E, k, gating, eps, inv_rms, logits,
                                       idx, gates, s, nullptr);
}

}  // namespace

cudaError_t launch_router(const void *x, const void *Wg, const float *bias, int T, int d, int E,
                          int k, int dt, int gating, float eps, float *inv_rms, float *logits,
                          int *idx, float *gates, cudaStream_t s, void *x_copy) {
    if (T == 0) return cudaSuccess;
    if (dt == MOE_BF16)
        return router_dispatch<__nv_bfloat16>(x, Wg, bias, T, d, E, k, gating, eps, inv_rms,
                                              logits, idx, gates, s, x_copy);
    return router_dispatch<float>(x, Wg, bias, T, d, E, k, gating, eps, inv_rms, logits, idx,
                                  gates, s, x_copy);
}

bool router_reads_host_rows(int T, int E) { return E <= 8 && T < 1536; }

cudaError_t launch_topk_from_logits(const float *logits, int T, int E, int k, int gating,
                                    int *idx, float *gates, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    return launch_pdl(topk_kernel, (T + 127) / 128, 128, 0, s, logits, T, E, k, gating, idx,
                      gates);
}

}  // namespace moe
