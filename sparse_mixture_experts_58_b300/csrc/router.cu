// Router: logits = x . W_g (fp32 accumulation), top-k selection (k <= 2,
// ties to the lower expert index) and the softmax over the kept logits
// ("Mixtral of Experts" (azimuth.plus), router paragraph).  Also counts, per
// chunk of kChunk tokens, how many rows each expert receives; the grouping
// pass turns those counts into row positions.
//
// HBM-bound: it reads x once (T*d elements) and W_g from L1/L2.  One warp
// handles two tokens at a time so each W_g vector fetched is used twice.
#include "internal.h"

namespace moe {
namespace {

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ void unpack4f(const uint4 &v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
}

template <typename T> struct Vec;
template <> struct Vec<__nv_bfloat16> {
    static constexpr int n = 8;
    __device__ static void unpack(const uint4 &v, float (&f)[8]) { unpack8(v, f); }
};
template <> struct Vec<float> {
    static constexpr int n = 4;
    __device__ static void unpack(const uint4 &v, float (&f)[4]) { unpack4f(v, f); }
};

// Finish one token: bias, top-k, gates, outputs, chunk count.
template <int EMAX>
__device__ __forceinline__ void finish_token(const float (&acc)[EMAX], const float *bias, int t,
                                             int E, int k, float *logits, int *idx, float *gates,
                                             int *s_cnt) {
    float l[EMAX];
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        if (e < E) {
            l[e] = acc[e] + (bias != nullptr ? bias[e] : 0.f);
            logits[(size_t)t * E + e] = l[e];
        }
    }
    int sel[2];
    float g[2];
    top2_gates(l, E, k, sel, g);
    for (int j = 0; j < k; ++j) {
        idx[(size_t)t * k + j] = sel[j];
        gates[(size_t)t * k + j] = g[j];
        atomicAdd(&s_cnt[sel[j]], 1);
    }
}

// One block = one chunk of kChunk tokens: 8 warps x 2 tokens.
template <typename T, int EMAX>
__global__ void __launch_bounds__(256) router_kernel(const T *__restrict__ x,
                                                     const T *__restrict__ Wg,
                                                     const float *__restrict__ bias, int Tn,
                                                     int d, int E, int k, float *logits, int *idx,
                                                     float *gates, int *chunk_counts) {
    constexpr int VN = Vec<T>::n;
    __shared__ int s_cnt[EMAX];
    if (threadIdx.x < EMAX) s_cnt[threadIdx.x] = 0;
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * kChunk + warp * 2;
    const bool has0 = t0 < Tn, has1 = t0 + 1 < Tn;
    float acc0[EMAX], acc1[EMAX];
#pragma unroll
    for (int e = 0; e < EMAX; ++e) acc0[e] = acc1[e] = 0.f;

    const int nvec = d / VN;
    const uint4 *xr0 = reinterpret_cast<const uint4 *>(x + (size_t)t0 * d);
    const uint4 *xr1 = reinterpret_cast<const uint4 *>(x + (size_t)(t0 + 1) * d);
    const uint4 zero = make_uint4(0, 0, 0, 0);
    if (has0) {
#pragma unroll 2
        for (int v = lane; v < nvec; v += 32) {
            float a[VN], b[VN];
            Vec<T>::unpack(__ldcs(xr0 + v), a);
            Vec<T>::unpack(has1 ? __ldcs(xr1 + v) : zero, b);
#pragma unroll
            for (int e = 0; e < EMAX; ++e) {
                if (e < E) {
                    float w[VN];
                    Vec<T>::unpack(__ldg(reinterpret_cast<const uint4 *>(Wg + (size_t)e * d) + v),
                                   w);
#pragma unroll
                    for (int i = 0; i < VN; ++i) {
                        acc0[e] = fmaf(a[i], w[i], acc0[e]);
                        acc1[e] = fmaf(b[i], w[i], acc1[e]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            acc0[e] += __shfl_xor_sync(0xffffffffu, acc0[e], off);
            acc1[e] += __shfl_xor_sync(0xffffffffu, acc1[e], off);
        }
    }
    if (lane == 0 && has0) finish_token<EMAX>(acc0, bias, t0, E, k, logits, idx, gates, s_cnt);
    if (lane == 1 && has1) finish_token<EMAX>(acc1, bias, t0 + 1, E, k, logits, idx, gates, s_cnt);
    __syncthreads();
    if (chunk_counts != nullptr && threadIdx.x < E)
        chunk_counts[(size_t)blockIdx.x * E + threadIdx.x] = s_cnt[threadIdx.x];
}

// Selection from given logits: one thread per token, 128 tokens (8 chunks)
// per block.
template <int EMAX>
__global__ void __launch_bounds__(128) topk_kernel(const float *__restrict__ logits, int Tn, int E,
                                                   int k, int *idx, float *gates,
                                                   int *chunk_counts, int nchunks) {
    constexpr int CPB = 128 / kChunk;
    __shared__ int s_cnt[CPB][EMAX];
    for (int i = threadIdx.x; i < CPB * EMAX; i += blockDim.x) (&s_cnt[0][0])[i] = 0;
    __syncthreads();
    const int t = blockIdx.x * 128 + threadIdx.x;
    if (t < Tn) {
        float l[EMAX];
#pragma unroll
        for (int e = 0; e < EMAX; ++e)
            if (e < E) l[e] = logits[(size_t)t * E + e];
        int sel[2];
        float g[2];
        top2_gates(l, E, k, sel, g);
        for (int j = 0; j < k; ++j) {
            idx[(size_t)t * k + j] = sel[j];
            gates[(size_t)t * k + j] = g[j];
            atomicAdd(&s_cnt[threadIdx.x / kChunk][sel[j]], 1);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < CPB * E; i += blockDim.x) {
        const int c = blockIdx.x * CPB + i / E;
        if (c < nchunks) chunk_counts[(size_t)c * E + i % E] = s_cnt[i / E][i % E];
    }
}

template <typename T>
cudaError_t router_dispatch(const void *x, const void *Wg, const float *bias, int T_, int d,
                            int E, int k, float *logits, int *idx, float *gates, int *cc,
                            cudaStream_t s) {
    const int nchunks = (T_ + kChunk - 1) / kChunk;
    const T *xp = static_cast<const T *>(x);
    const T *wp = static_cast<const T *>(Wg);
    if (E <= 8)
        router_kernel<T, 8><<<nchunks, 256, 0, s>>>(xp, wp, bias, T_, d, E, k, logits, idx, gates, cc);
    else if (E <= 16)
        router_kernel<T, 16><<<nchunks, 256, 0, s>>>(xp, wp, bias, T_, d, E, k, logits, idx, gates, cc);
    else
        router_kernel<T, 32><<<nchunks, 256, 0, s>>>(xp, wp, bias, T_, d, E, k, logits, idx, gates, cc);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const void *x, const void *Wg, const float *bias, int T, int d, int E,
                          int k, int dt, float *logits, int *idx, float *gates, int *chunk_counts,
                          cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (dt == MOE_BF16)
        return router_dispatch<__nv_bfloat16>(x, Wg, bias, T, d, E, k, logits, idx, gates,
                                              chunk_counts, s);
    return router_dispatch<float>(x, Wg, bias, T, d, E, k, logits, idx, gates, chunk_counts, s);
}

cudaError_t launch_topk_from_logits(const float *logits, int T, int E, int k, int *idx,
                                    float *gates, int *chunk_counts, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int nchunks = (T + kChunk - 1) / kChunk;
    const int grid = (T + 127) / 128;
    if (E <= 8)
        topk_kernel<8><<<grid, 128, 0, s>>>(logits, T, E, k, idx, gates, chunk_counts, nchunks);
    else if (E <= 16)
        topk_kernel<16><<<grid, 128, 0, s>>>(logits, T, E, k, idx, gates, chunk_counts, nchunks);
    else
        topk_kernel<32><<<grid, 128, 0, s>>>(logits, T, E, k, idx, gates, chunk_counts, nchunks);
    return cudaGetLastError();
}

}  // namespace moe
