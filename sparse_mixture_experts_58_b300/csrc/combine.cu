// Gated combine back to token order, plus the stacked-layer RMSNorm/residual
// helper and the bounded-wait self-test kernel.
//
// Combine: out[t] = sum_j gates[t][j] * y_{row(t,j)}, the selected experts'
// outputs weighted by the routing weights ("Mixtral & Sparse MoE (2024) > The
// Solution", routing paragraph; "Mixtral" curriculum page, "weighted expert
// outputs").  The down projection leaves fp32 partial sums per contraction
// split; they are added here in split order, then gated in slot order, then
// rounded once.  HBM-bound: one warp per token, 16-byte loads.  In a
// pre-norm block the residual add follows in the same pass:
// out <- round(out + round(combined)), the rounding the separate add would do.
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

template <typename T>
__device__ __forceinline__ void store4(T *p, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float *p, float4 v) {
    *reinterpret_cast<float4 *>(p) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *p, float4 v) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t *>(&a);
    u.y = *reinterpret_cast<const uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
}

template <typename T>
__device__ __forceinline__ float4 load4(const T *p);
template <>
__device__ __forceinline__ float4 load4<float>(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}

template <typename T>
__device__ __forceinline__ float round_to(float v) {
    return to_f32(from_f32<T>(v));
}

__device__ __forceinline__ void add4(float4 &s, const float4 &p) {
    s.x += p.x;
    s.y += p.y;
    s.z += p.z;
    s.w += p.w;
}

// Block (t, c): token t, columns [4 * C * 256 c, ...): each thread owns C
// groups of four columns, 256 groups apart.  For each of the token's k <= K
// slots, up to SB split partials of all C groups are loaded together, then
// added in split order, so a thread has K * C * SB loads in flight per round
// trip.  A slot with inv < 0 was dropped by a capacity limit and contributes
// nothing; with `renorm` the kept gates are scaled by (sum of all the token's
// gates) / (sum of its kept gates), and a token with no kept slot gets 0.
template <typename T, int K, int C, int SB>
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ y, int splits,
                                                      int rows, const float *__restrict__ gates,
                                                      const int *__restrict__ inv, int Tn, int d,
                                                      int k, int renorm, int residual, T *out) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    const int nv = d / 4;
    const int v0 = blockIdx.y * 256 * C + threadIdx.x;  // first float4 column group
    const size_t stride4 = (size_t)rows * nv;            // one split, in float4
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    int rowj[K];
    float gj[K];
    bool use[K];
    float total = 0.f, kept_total = 0.f;
#pragma unroll
    for (int j = 0; j < K; ++j) {
        rowj[j] = 0;
        gj[j] = 0.f;
        use[j] = false;
        if (j < k) {
            const int r = inv[(size_t)t * k + j];
            gj[j] = gates[(size_t)t * k + j];
            total += gj[j];
            use[j] = r >= 0;
            if (use[j]) {
                rowj[j] = r;
                kept_total += gj[j];
            }
        }
    }
    if (renorm) {
        const float f = kept_total > 0.f ? total / kept_total : 0.f;
#pragma unroll
        for (int j = 0; j < K; ++j) gj[j] *= f;
    }
    float4 s[K][C];
    for (int q0 = 0; q0 < splits; q0 += SB) {
        float4 p[K][C][SB];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const float4 *src = reinterpret_cast<const float4 *>(y) + (size_t)rowj[j] * nv;
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const int v = v0 + 256 * c;
#pragma unroll
                for (int i = 0; i < SB; ++i)
                    p[j][c][i] = (use[j] && v < nv && q0 + i < splits)
                                     ? __ldcs(src + (size_t)(q0 + i) * stride4 + v)
                                     : zero;
            }
        }
#pragma unroll
        for (int j = 0; j < K; ++j) {
#pragma unroll
            for (int c = 0; c < C; ++c) {
                if (q0 == 0) s[j][c] = p[j][c][0];
                else add4(s[j][c], p[j][c][0]);
#pragma unroll
                for (int i = 1; i < SB; ++i)
                    if (q0 + i < splits) add4(s[j][c], p[j][c][i]);
            }
        }
    }
#pragma unroll
    for (int c = 0; c < C; ++c) {
        const int v = v0 + 256 * c;
        if (v >= nv) continue;
        float4 acc = zero;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (use[j]) {
                acc.x = fmaf(gj[j], s[j][c].x, acc.x);
                acc.y = fmaf(gj[j], s[j][c].y, acc.y);
                acc.z = fmaf(gj[j], s[j][c].z, acc.z);
                acc.w = fmaf(gj[j], s[j][c].w, acc.w);
            }
        }
        T *dst = out + (size_t)t * d + 4 * v;
        if (residual) {
            const float4 r = load4<T>(dst);
            acc = make_float4(r.x + round_to<T>(acc.x), r.y + round_to<T>(acc.y),
                              r.z + round_to<T>(acc.z), r.w + round_to<T>(acc.w));
        }
        store4<T>(dst, acc);
    }
}

template <typename T, int K, int C, int SB>
void launch_combine_t(const float *y, int splits, int rows, const float *gates, const int *inv,
                      int T_, int d, int k, int renorm, int residual, void *out, cudaStream_t s) {
    const dim3 grid(T_, (d / 4 + 256 * C - 1) / (256 * C));
    launch_pdl(combine_kernel<T, K, C, SB>, grid, 256, 0, s, y, splits, rows, gates, inv, T_, d, k,
               renorm, residual, static_cast<T *>(out));
}

// Kernel shape by slot count and split count, keeping about 16 loads in
// flight per thread: unsplit or lightly split partials (large batches) take
// 2-4 column groups per thread; heavily split partials (small batches) one
// group and up to 8 splits per batch.
template <typename T>
void launch_combine_dt(const float *y, int splits, int rows, const float *gates, const int *inv,
                       int T_, int d, int k, int renorm, int residual, void *out, cudaStream_t s) {
    void (*launch)(const float *, int, int, const float *, const int *, int, int, int, int, int,
                   void *, cudaStream_t);
    if (k <= 2) {
        if (splits == 1)
            launch = launch_combine_t<T, 2, 4, 1>;
        else if (splits == 2)
            launch = launch_combine_t<T, 2, 4, 2>;
        else if (splits <= 4)
            launch = launch_combine_t<T, 2, 2, 4>;
        else
            launch = launch_combine_t<T, 2, 1, 8>;
    } else {
        launch = splits == 1 ? launch_combine_t<T, MOE_MAX_TOPK, 1, 1>
                             : launch_combine_t<T, MOE_MAX_TOPK, 1, 2>;
    }
    launch(y, splits, rows, gates, inv, T_, d, k, renorm, residual, out, s);
}

// Gated sums accumulated by the down projection's epilogue (fp32 [T][d], the
// gate-weighted outputs of a token's slots added into a zeroed row) rounded
// once to the output type; with `residual`, out <- round(out + round(sum)),
// the rounding of the combine's residual form.  One block per (token, 1024 * C
// columns), 16-byte loads.
template <typename T, int C>
__global__ void __launch_bounds__(256) finalize_kernel(const float *__restrict__ acc, int d,
                                                       int residual, T *out) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    const int nv = d / 4;
    const float4 *src = reinterpret_cast<const float4 *>(acc) + (size_t)t * nv;
    float4 a[C];
#pragma unroll
    for (int c = 0; c < C; ++c) {
        const int v = blockIdx.y * 256 * C + threadIdx.x + 256 * c;
        a[c] = v < nv ? __ldcs(src + v) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int c = 0; c < C; ++c) {
        const int v = blockIdx.y * 256 * C + threadIdx.x + 256 * c;
        if (v >= nv) continue;
        T *dst = out + (size_t)t * d + 4 * v;
        float4 o = a[c];
        if (residual) {
            const float4 r = load4<T>(dst);
            o = make_float4(r.x + round_to<T>(o.x), r.y + round_to<T>(o.y),
                            r.z + round_to<T>(o.z), r.w + round_to<T>(o.w));
        }
        store4<T>(dst, o);
    }
}

// One block of kNormThreads per row: optional residual add (rounded to the
// storage type), then RMSNorm with gain 1 in the order common.cuh fixes, the
// order the router's fused normalisation repeats.  d is a multiple of one
// 16-byte slice.
template <typename T>
__global__ void __launch_bounds__(kNormThreads)
    add_rmsnorm_kernel(T *x, const T *__restrict__ add, T *xn, int d, float eps) {
    constexpr int VN = Vec<T>::n;
    __shared__ float s_part[kNormThreads / 32];
    pdl_wait();
    pdl_trigger();
    const size_t o = (size_t)blockIdx.x * d;
    uint4 *xr = reinterpret_cast<uint4 *>(x + o);
    const uint4 *ar = add != nullptr ? reinterpret_cast<const uint4 *>(add + o) : nullptr;
    uint4 *xnr = reinterpret_cast<uint4 *>(xn + o);
    const int nvec = d / VN;
    float ss = 0.f;
    for (int v = threadIdx.x; v < nvec; v += kNormThreads) {
        uint4 q = xr[v];
        if (ar != nullptr) {
            float a[VN], b[VN];
            Vec<T>::unpack(q, a);
            Vec<T>::unpack(ar[v], b);
#pragma unroll
            for (int i = 0; i < VN; ++i) a[i] += b[i];
            q = Vec<T>::pack(a);
            xr[v] = q;
        }
        ss = slice_sumsq<T>(ss, q);
    }
    ss = warp_butterfly_sum(ss);
    if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) tot += s_part[w];
    const float scale = rms_scale(tot, d, eps);
    for (int v = threadIdx.x; v < nvec; v += kNormThreads) xnr[v] = scale_slice<T>(xr[v], scale);
}

// Waits on a barrier nothing arrives at; the bounded wait gives up after
// `limit_ns` and records kStatusSelftest.
__global__ void wait_selftest_kernel(unsigned long long limit_ns, int *status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::fence_barrier_init();
        ptx::mbar_wait_bounded(&bar, 0, nullptr, status, kStatusSelftest, limit_ns);
    }
}

}  // namespace

cudaError_t launch_combine(const float *y, int splits, int rows, const float *gates,
                           const int *inv, int T, int d, int k, int renorm, int residual, int dt,
                           void *out, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (dt == MOE_BF16)
        launch_combine_dt<__nv_bfloat16>(y, splits, rows, gates, inv, T, d, k, renorm, residual,
                                         out, s);
    else
        launch_combine_dt<float>(y, splits, rows, gates, inv, T, d, k, renorm, residual, out, s);
    return cudaGetLastError();
}

cudaError_t launch_finalize(const float *acc, int T, int d, int residual, int dt, void *out,
                            cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    constexpr int C = 2;
    const dim3 grid(T, (d / 4 + 256 * C - 1) / (256 * C));
    if (dt == MOE_BF16)
        return launch_pdl(finalize_kernel<__nv_bfloat16, C>, grid, 256, 0, s, acc, d, residual,
                          static_cast<__nv_bfloat16 *>(out));
    return launch_pdl(finalize_kernel<float, C>, grid, 256, 0, s, acc, d, residual,
                      static_cast<float *>(out));
}

cudaError_t launch_add_rmsnorm(void *x, const void *add, void *xn, int T, int d, float eps, int dt,
                               cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (dt == MOE_BF16)
        return launch_pdl(add_rmsnorm_kernel<__nv_bfloat16>, T, kNormThreads, 0, s,
                          static_cast<__nv_bfloat16 *>(x),
                          static_cast<const __nv_bfloat16 *>(add),
                          static_cast<__nv_bfloat16 *>(xn), d, eps);
    return launch_pdl(add_rmsnorm_kernel<float>, T, kNormThreads, 0, s, static_cast<float *>(x),
                      static_cast<const float *>(add), static_cast<float *>(xn), d, eps);
}

cudaError_t launch_wait_selftest(unsigned int limit_ns, cudaStream_t s) {
    int *st = device_status_ptr();
    if (st == nullptr) return cudaErrorUnknown;
    wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, st);
    return cudaGetLastError();
}

}  // namespace moe
