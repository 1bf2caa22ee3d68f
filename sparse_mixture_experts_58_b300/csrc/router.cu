// Router: logits = x . W_g (fp32 accumulation), top-k selection (k <= 2,
// ties to the lower expert index) and the softmax over the kept logits
// ("Mixtral of Experts" (azimuth.plus), router paragraph).
//
// One block handles two tokens.  Its 256 threads split the hidden dimension:
// each thread takes 16-byte slices of both token rows and the same slices of
// every expert's router row, issues all of those loads before any arithmetic
// (one memory round trip when d <= 256 slices per thread pass), then the block
// reduces the per-thread partial sums in a fixed order.  HBM traffic is x
// once; the 64 KB router matrix is served from L1/L2.
//
// Fused RMSNorm (pre-norm blocks): a first pass over the two rows gives each
// token's RMSNorm scale (stored for the grouping pass); the logits are then
// taken of round(x * scale), the normalised row the stand-alone RMSNorm
// kernel would have stored, read again from L1.
#include "internal.h"

namespace moe {
namespace {

constexpr int kRouterThreads = kNormThreads;
constexpr int kRouterTokens = 2;

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
template <typename T, int EG, int V, bool NORM>
__global__ void __launch_bounds__(kRouterThreads) router_kernel(
    const T *__restrict__ x, const T *__restrict__ Wg, const float *__restrict__ bias, int Tn,
    int d, int E, int k, int gating, float eps, float *inv_rms, float *logits, int *idx,
    float *gates) {
    constexpr int VN = Vec<T>::n;
    constexpr int NW = kRouterThreads / 32;
    __shared__ float s_part[NW][kRouterTokens][MOE_MAX_EXPERTS];
    __shared__ float s_l[kRouterTokens][MOE_MAX_EXPERTS];
    __shared__ float s_ss[NW][kRouterTokens];
    __shared__ float s_scale[kRouterTokens];

    pdl_wait();
    pdl_trigger();
    const int t0 = blockIdx.x * kRouterTokens;
    const bool has1 = t0 + 1 < Tn;
    const int nvec = d / VN;
    const uint4 *xr0 = reinterpret_cast<const uint4 *>(x + (size_t)t0 * d);
    const uint4 *xr1 = reinterpret_cast<const uint4 *>(x + (size_t)(has1 ? t0 + 1 : t0) * d);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    float sc0 = 1.f, sc1 = 1.f;
    if (NORM) {
        float ss0 = 0.f, ss1 = 0.f;
        for (int v = threadIdx.x; v < nvec; v += kRouterThreads) {
            ss0 = slice_sumsq<T>(ss0, xr0[v]);
            ss1 = slice_sumsq<T>(ss1, xr1[v]);
        }
        ss0 = warp_butterfly_sum(ss0);
        ss1 = warp_butterfly_sum(ss1);
        if (lane == 0) {
            s_ss[warp][0] = ss0;
            s_ss[warp][1] = ss1;
        }
        __syncthreads();
        if (threadIdx.x < kRouterTokens) {
            float tot = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < NW; ++w2) tot += s_ss[w2][threadIdx.x];
            const float sc = rms_scale(tot, d, eps);
            s_scale[threadIdx.x] = sc;
            if (t0 + (int)threadIdx.x < Tn) inv_rms[t0 + threadIdx.x] = sc;
        }
        __syncthreads();
        sc0 = s_scale[0];
        sc1 = s_scale[1];
    }

    for (int g0 = 0; g0 < E; g0 += EG) {
        const uint4 *wr[EG];
#pragma unroll
        for (int e = 0; e < EG; ++e)
            wr[e] = reinterpret_cast<const uint4 *>(Wg + (size_t)(g0 + e < E ? g0 + e : E - 1) * d);
        float acc0[EG], acc1[EG];
#pragma unroll
        for (int e = 0; e < EG; ++e) acc0[e] = acc1[e] = 0.f;
        for (int v0 = threadIdx.x; v0 < nvec; v0 += kRouterThreads * V) {
            uint4 xa[V], xb[V], w[V][EG];
#pragma unroll
            for (int u = 0; u < V; ++u) {
                const int v = v0 + kRouterThreads * u;
                const int vv = v < nvec ? v : 0;
                xa[u] = __ldcs(xr0 + vv);
                xb[u] = __ldcs(xr1 + vv);
#pragma unroll
                for (int e = 0; e < EG; ++e) w[u][e] = __ldg(wr[e] + vv);
                if (v >= nvec) xa[u] = xb[u] = zero;
            }
#pragma unroll
            for (int u = 0; u < V; ++u) {
                float a[VN], b[VN];
                Vec<T>::unpack(NORM ? scale_slice<T>(xa[u], sc0) : xa[u], a);
                Vec<T>::unpack(NORM ? scale_slice<T>(xb[u], sc1) : xb[u], b);
#pragma unroll
                for (int e = 0; e < EG; ++e) {
                    float wf[VN];
                    Vec<T>::unpack(w[u][e], wf);
#pragma unroll
                    for (int i = 0; i < VN; ++i) {
                        acc0[e] = fmaf(a[i], wf[i], acc0[e]);
                        acc1[e] = fmaf(b[i], wf[i], acc1[e]);
                    }
                }
            }
        }
        // butterfly within each warp; lane 0 parks the warp's sums
#pragma unroll
        for (int e = 0; e < EG; ++e) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                acc0[e] += __shfl_xor_sync(0xffffffffu, acc0[e], off);
                acc1[e] += __shfl_xor_sync(0xffffffffu, acc1[e], off);
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int e = 0; e < EG; ++e) {
                if (g0 + e < E) {
                    s_part[warp][0][g0 + e] = acc0[e];
                    s_part[warp][1][g0 + e] = acc1[e];
                }
            }
        }
    }
    __syncthreads();
    // warps added in order: one thread per (token, expert)
    for (int i = threadIdx.x; i < kRouterTokens * E; i += kRouterThreads) {
        const int j = i / E, e = i - j * E;
        float s = s_part[0][j][e];
#pragma unroll
        for (int w2 = 1; w2 < NW; ++w2) s += s_part[w2][j][e];
        s_l[j][e] = s;
    }
    __syncthreads();
    if (threadIdx.x < kRouterTokens && (threadIdx.x == 0 || has1))
        finish_token(s_l[threadIdx.x], bias, t0 + threadIdx.x, E, k, gating, logits, idx, gates);
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

template <typename T, bool NORM>
cudaError_t router_dispatch_n(const void *x, const void *Wg, const float *bias, int T_, int d,
                              int E, int k, int gating, float eps, float *inv_rms, float *logits,
                              int *idx, float *gates, cudaStream_t s) {
    const int grid = (T_ + kRouterTokens - 1) / kRouterTokens;
    const T *xp = static_cast<const T *>(x);
    const T *wp = static_cast<const T *>(Wg);
    // 16-byte loads in flight per thread per pass: V * (2 + EG)
    if (E <= 8)
        return launch_pdl(router_kernel<T, 8, 2, NORM>, grid, kRouterThreads, 0, s, xp, wp, bias,
                          T_, d, E, k, gating, eps, inv_rms, logits, idx, gates);
    return launch_pdl(router_kernel<T, 16, 1, NORM>, grid, kRouterThreads, 0, s, xp, wp, bias, T_,
                      d, E, k, gating, eps, inv_rms, logits, idx, gates);
}

template <typename T>
cudaError_t router_dispatch(const void *x, const void *Wg, const float *bias, int T_, int d,
                            int E, int k, int gating, float eps, float *inv_rms, float *logits,
                            int *idx, float *gates, cudaStream_t s) {
    if (inv_rms != nullptr)
        return router_dispatch_n<T, true>(x, Wg, bias, T_, d, E, k, gating, eps, inv_rms, logits,
                                          idx, gates, s);
    return router_dispatch_n<T, false>(x, Wg, bias, T_, d, E, k, gating, eps, inv_rms, logits,
                                       idx, gates, s);
}

}  // namespace

cudaError_t launch_router(const void *x, const void *Wg, const float *bias, int T, int d, int E,
                          int k, int dt, int gating, float eps, float *inv_rms, float *logits,
                          int *idx, float *gates, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (dt == MOE_BF16)
        return router_dispatch<__nv_bfloat16>(x, Wg, bias, T, d, E, k, gating, eps, inv_rms,
                                              logits, idx, gates, s);
    return router_dispatch<float>(x, Wg, bias, T, d, E, k, gating, eps, inv_rms, logits, idx,
                                  gates, s);
}

cudaError_t launch_topk_from_logits(const float *logits, int T, int E, int k, int gating,
                                    int *idx, float *gates, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    return launch_pdl(topk_kernel, (T + 127) / 128, 128, 0, s, logits, T, E, k, gating, idx,
                      gates);
}

}  // namespace moe
