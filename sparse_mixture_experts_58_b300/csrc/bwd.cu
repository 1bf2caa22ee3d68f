// Backward of the layer outside the expert GEMMs: gathering rows into the
// padded expert grouping, the router's backward and the input gradient.
//
// With g the kept gates of a token (a softmax over its k kept logits: "Mixtral
// of Experts" (azimuth.plus), router paragraph) and dg_j = <dout[t], y_j> the
// gradient of the loss with respect to gate j, the kept logits receive
//   dl_j = g_j (dg_j - sum_m g_m dg_m),
// the router matrix dW_g[e] = sum over tokens of dl_j x[t] (e = e_j), and the
// token's input gradient adds sum_j dl_j W_g[e_j] to the experts' part
// sum_j dX[row_j].  Every sum runs in a fixed order, so the results do not
// depend on scheduling.
#include "internal.h"

namespace moe {
namespace {

// One warp per row: dst[r] = src[perm[r] / k] (zeros for a padding row,
// perm[r] < 0), for r < offsets[E]; optional row_gate[r] = gates[perm[r]].
__global__ void __launch_bounds__(256) gather_rows_kernel(
    const uint4 *__restrict__ src, const int *__restrict__ perm, const int *__restrict__ offsets,
    int E, int rows, int k, int rowvec, const float *__restrict__ gates, float *row_gate,
    uint4 *dst) {
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows || r >= offsets[E]) return;
    const int p = perm[r];
    if (row_gate != nullptr && lane == 0) row_gate[r] = p >= 0 ? gates[p] : 0.f;
    uint4 *d = dst + (size_t)r * rowvec;
    if (p < 0) {
        for (int v = lane; v < rowvec; v += 32) d[v] = make_uint4(0, 0, 0, 0);
        return;
    }
    const uint4 *s = src + (size_t)(p / k) * rowvec;
    constexpr int U = 4;
    for (int v0 = lane; v0 < rowvec; v0 += 32 * U) {
        uint4 val[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + 32 * u;
            val[u] = v < rowvec ? __ldg(s + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v0 + 32 * u < rowvec) d[v0 + 32 * u] = val[u];
    }
}

// Block-wide sum in a fixed order (butterfly in each warp, then the warps in
// order); every thread gets the result.
__device__ __forceinline__ float block_sum(float v, float *s_part) {
    v = warp_butterfly_sum(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += s_part[w];
    return t;
}

// One block per token.
__global__ void __launch_bounds__(256) router_bwd_kernel(
    const int *__restrict__ idx, const float *__restrict__ gates, const int *__restrict__ inv,
    const float *__restrict__ dgp, int nblk, const float *__restrict__ dx_rows,
    const __nv_bfloat16 *__restrict__ Wg, int d, int k, float *dl, __nv_bfloat16 *dx) {
    __shared__ float s_part[8];
    __shared__ float s_dl[MOE_MAX_TOPK];
    __shared__ int s_row[MOE_MAX_TOPK], s_e[MOE_MAX_TOPK];
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    float dg[MOE_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j) {
        dg[j] = 0.f;
        if (j < k) {
            const int row = inv[(size_t)t * k + j];
            float p = 0.f;
            for (int b = threadIdx.x; b < nblk; b += blockDim.x) p += dgp[(size_t)row * nblk + b];
            dg[j] = block_sum(p, s_part);
        }
    }
    if (threadIdx.x == 0) {
        float gdg = 0.f;
        for (int j = 0; j < k; ++j) gdg += gates[(size_t)t * k + j] * dg[j];
        for (int j = 0; j < k; ++j) {
            const float g = gates[(size_t)t * k + j];
            s_dl[j] = g * (dg[j] - gdg);
            dl[(size_t)t * k + j] = s_dl[j];
            s_row[j] = inv[(size_t)t * k + j];
            s_e[j] = idx[(size_t)t * k + j];
        }
    }
    __syncthreads();
    for (int i = threadIdx.x * 2; i < d; i += blockDim.x * 2) {
        float a0 = 0.f, a1 = 0.f;
        for (int j = 0; j < k; ++j) {
            const float2 v = *reinterpret_cast<const float2 *>(dx_rows + (size_t)s_row[j] * d + i);
            a0 += v.x;
            a1 += v.y;
        }
        for (int j = 0; j < k; ++j) {
            const __nv_bfloat162 w =
                *reinterpret_cast<const __nv_bfloat162 *>(Wg + (size_t)s_e[j] * d + i);
            a0 = fmaf(s_dl[j], __low2float(w), a0);
            a1 = fmaf(s_dl[j], __high2float(w), a1);
        }
        *reinterpret_cast<__nv_bfloat162 *>(dx + (size_t)t * d + i) = __floats2bfloat162_rn(a0, a1);
    }
}

// Router-matrix gradient, first pass: block (column chunk, token slice)
// accumulates, for every expert, dl * x over its slice's tokens in order.
constexpr int kWgThreads = 128;
constexpr int kWgTokens = 64;

template <int EREG>
__global__ void __launch_bounds__(kWgThreads) router_wgrad_part_kernel(
    const int *__restrict__ idx, const float *__restrict__ dl,
    const __nv_bfloat16 *__restrict__ x, int T, int d, int E, int k, float *part) {
    // The slice's expert ids and logit gradients are staged in shared memory
    // first, so the token loop waits on x only.  EREG > 0 (E <= EREG): one
    // register accumulator per expert, each selection added with a compare
    // and select; otherwise accumulators in shared memory.
    __shared__ float s_acc[EREG > 0 ? 1 : MOE_MAX_EXPERTS][kWgThreads];
    __shared__ int s_e[kWgTokens * 4];
    __shared__ float s_g[kWgTokens * 4];
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x * kWgThreads + threadIdx.x;
    const int slice = blockIdx.y;
    float acc[EREG > 0 ? EREG : 1];
#pragma unroll
    for (int e = 0; e < (EREG > 0 ? EREG : 1); ++e) acc[e] = 0.f;
    if (EREG == 0)
        for (int e = 0; e < E; ++e) s_acc[e][threadIdx.x] = 0.f;
    const int t_first = slice * kWgTokens;
    const int t1 = min(T, t_first + kWgTokens);
    const int tstep = (kWgTokens * 4) / k;  // tokens per staging round (k <= 8)
    for (int ts = t_first; ts < t1; ts += tstep) {
        const int te = min(t1, ts + tstep);
        __syncthreads();
        for (int q = threadIdx.x; q < (te - ts) * k; q += kWgThreads) {
            s_e[q] = idx[(size_t)ts * k + q];
            s_g[q] = dl[(size_t)ts * k + q];
        }
        __syncthreads();
        if (i < d) {
#pragma unroll 4
            for (int t = ts; t < te; ++t) {
                const float xv = __bfloat162float(x[(size_t)t * d + i]);
                for (int j = 0; j < k; ++j) {
                    const int q = (t - ts) * k + j;
                    const int e = s_e[q];
                    const float gx = s_g[q] * xv;
                    if (EREG > 0) {
#pragma unroll
                        for (int r = 0; r < (EREG > 0 ? EREG : 1); ++r) acc[r] += (e == r) ? gx : 0.f;
                    } else {
                        s_acc[e][threadIdx.x] += gx;
                    }
                }
            }
        }
    }
    if (i < d)
        for (int e = 0; e < E; ++e)
            part[((size_t)slice * E + e) * d + i] = EREG > 0 ? acc[e < EREG ? e : 0] : s_acc[e][threadIdx.x];
}

// Second pass: dWg[e][i] = sum of the slices' partial sums in slice order.
__global__ void __launch_bounds__(256) router_wgrad_sum_kernel(const float *__restrict__ part,
                                                               int slices, int E, int d,
                                                               float *dWg) {
    pdl_wait();
    pdl_trigger();
    const size_t n = (size_t)E * d;
    const size_t o = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (o >= n) return;
    float s = 0.f;
    for (int q = 0; q < slices; ++q) s += part[(size_t)q * n + o];
    dWg[o] = s;
}

}  // namespace

cudaError_t launch_gather_rows(const void *src, const int *perm, const int *offsets, int E,
                               int rows, int k, int d, const float *gates, float *row_gate,
                               void *dst, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const int rowvec = d * 2 / 16;
    return launch_pdl(gather_rows_kernel, (rows + 7) / 8, 256, 0, s,
                      static_cast<const uint4 *>(src), perm, offsets, E, rows, k, rowvec, gates,
                      row_gate, static_cast<uint4 *>(dst));
}

cudaError_t launch_router_bwd(const int *idx, const float *gates, const int *inv,
                              const float *dgp, int nblk, const float *dx_rows, const void *Wg,
                              int T, int d, int k, float *dl, void *dx, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    return launch_pdl(router_bwd_kernel, T, 256, 0, s, idx, gates, inv, dgp, nblk, dx_rows,
                      static_cast<const __nv_bfloat16 *>(Wg), d, k, dl,
                      static_cast<__nv_bfloat16 *>(dx));
}

size_t router_wg_part_floats(int T, int E, int d) {
    const size_t slices = (size_t)(T + kWgTokens - 1) / kWgTokens;
    return slices * E * d;
}

cudaError_t launch_router_wgrad(const int *idx, const float *dl, const void *x, int T, int d,
                                int E, int k, float *part, float *dWg, cudaStream_t s) {
    const int slices = (T + kWgTokens - 1) / kWgTokens;
    if (slices == 0) return cudaMemsetAsync(dWg, 0, sizeof(float) * E * d, s);
    const dim3 grid((d + kWgThreads - 1) / kWgThreads, slices);
    const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(x);
    cudaError_t e = E <= 8 ? launch_pdl(router_wgrad_part_kernel<8>, grid, kWgThreads, 0, s, idx,
                                        dl, xb, T, d, E, k, part)
                           : launch_pdl(router_wgrad_part_kernel<0>, grid, kWgThreads, 0, s, idx,
                                        dl, xb, T, d, E, k, part);
    if (e != cudaSuccess) return e;
    const size_t n = (size_t)E * d;
    return launch_pdl(router_wgrad_sum_kernel, (unsigned)((n + 255) / 256), 256, 0, s,
                      static_cast<const float *>(part), slices, E, d, dWg);
}

}  // namespace moe
