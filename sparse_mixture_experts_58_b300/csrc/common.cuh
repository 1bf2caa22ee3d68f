// Shared definitions for the libmoe kernels and host code.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Tokens per router chunk.  The router counts expert hits per chunk and the
// grouping pass ranks tokens inside a chunk, so both use this size.
constexpr int kChunk = 16;

// Rows of the contraction dimension per pipeline stage: 64 bf16 = 128 bytes,
// the width of one 128-byte-swizzled shared-memory row.
constexpr int kBlockK = 64;

// Default limit of every bounded wait inside a kernel (nanoseconds).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Codes written to the device status word when a bounded wait expires.
enum DeviceStatus : int {
    kStatusOk = 0,
    kStatusProducerWait = 1,   // TMA producer waited too long for a free stage
    kStatusMmaWait = 2,        // MMA issuer waited too long for data / accumulator
    kStatusEpilogueWait = 3,   // epilogue waited too long for an accumulator
    kStatusDrainWait = 4,      // teardown waited too long for in-flight work
    kStatusSelftest = 5        // the self-test wait expired (expected)
};

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch: every kernel of the layer is launched so it
// may start while the previous one finishes.  A kernel calls pdl_wait()
// before it touches anything an earlier kernel wrote (the wait returns once
// the previous grid has completed and its writes are visible), and then
// pdl_trigger() so the next kernel may be scheduled; since a kernel triggers
// only after its own wait returned, every kernel before it has completed too.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The first expired wait wins; later ones leave the word alone.
__device__ __forceinline__ void report_status(int *status, int code) {
    if (status != nullptr) atomicCAS(status, 0, code);
}

template <typename T> struct Elem;
template <> struct Elem<float> { static constexpr int size = 4; };
template <> struct Elem<__nv_bfloat16> { static constexpr int size = 2; };

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// 16-byte slices of a row: unpacked to fp32 in element order, and packed
// back with round-to-nearest-even to the storage type.
template <typename T> struct Vec;
template <> struct Vec<__nv_bfloat16> {
    static constexpr int n = 8;
    __device__ static void unpack(const uint4 &v, float (&f)[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    __device__ static uint4 pack(const float (&f)[8]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 p = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t *>(&p);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <> struct Vec<float> {
    static constexpr int n = 4;
    __device__ static void unpack(const uint4 &v, float (&f)[4]) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ static uint4 pack(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
};

// RMSNorm with gain 1, computed the same way (so to the same bits) by the
// stand-alone RMSNorm kernel and by the router's fused normalisation: with
// kNormThreads threads per row, thread i takes the row's 16-byte slices i,
// i + kNormThreads, ... and adds the squares of their elements in order
// (fmaf); each warp's partial sums are added by a butterfly, then the warps'
// sums in warp order; scale = 1 / sqrt(sum / d + eps); the normalised element
// is round(x * scale) in the storage type.
constexpr int kNormThreads = 256;

template <typename T>
__device__ __forceinline__ float slice_sumsq(float ss, const uint4 &v) {
    float f[Vec<T>::n];
    Vec<T>::unpack(v, f);
#pragma unroll
    for (int i = 0; i < Vec<T>::n; ++i) ss = fmaf(f[i], f[i], ss);
    return ss;
}

__device__ __forceinline__ float warp_butterfly_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// The butterfly sums of N values per lane at once (N a power of two <= 32),
// each lane keeping only some of them: at the step with offset o, while more
// than one value is left, a lane keeps the half of its values selected by
// (lane & o) and adds the partner lane's copy of that half, sending the other
// half; from then on the one value left is summed as in warp_butterfly_sum.
// Every sum is formed by the same additions, in the same order, as
// warp_butterfly_sum gives it (a + b == b + a), so the bits are the same; it
// costs N - 1 + (5 - log2 N) shuffles instead of 5 N.  On return v[0] holds
// the sum of value lane >> (5 - log2 N), in every lane.
template <int N>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[N], int lane) {
    static_assert(N >= 1 && N <= 32 && (N & (N - 1)) == 0, "N: a power of two up to 32");
    int off = 16;
#pragma unroll
    for (int n = N; n > 1; n >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? v[i] : v[i + n / 2];
            const float keep = upper ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
#pragma unroll
    for (; off > 0; off >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    return v[0];
}

__device__ __forceinline__ float rms_scale(float sumsq, int d, float eps) {
    return 1.f / sqrtf(sumsq / static_cast<float>(d) + eps);
}

// round(x * scale) for the elements of one 16-byte slice.
template <typename T>
__device__ __forceinline__ uint4 scale_slice(const uint4 &v, float scale) {
    float f[Vec<T>::n];
    Vec<T>::unpack(v, f);
#pragma unroll
    for (int i = 0; i < Vec<T>::n; ++i) f[i] *= scale;
    return Vec<T>::pack(f);
}

// Selection of the k (<= KMAX <= MOE_MAX_TOPK) largest of E logits: each
// logit in expert order is carried down a list of KMAX entries kept in
// (value descending, expert ascending) order, swapping places with any entry
// it precedes in that order -- a larger value, or an equal value of a lower
// expert (a displaced entry moving down can tie with the next one and must
// then stay ahead of it).  Slot 0 ends with the largest logit; equal logits
// keep ascending expert order.  Fully unrolled over the list: registers only.
// Gates, relative to the largest logit l0 so every exponent is <= 0:
//   gating 0: z_j = exp(l_j - l0), g_j = z_j / sum_j' z_j' (softmax over kept);
//   gating 1: g_j = exp(l_j - l0) / sum_e exp(l_e - l0) (full softmax, kept
//             entries not renormalised).
// The logits are read through `at(e)`; with EMAX > 0 the loops over experts
// are unrolled to EMAX (entries from E on ignored), so that logits held in a
// register array stay in registers.
template <int KMAX, int EMAX, typename At>
__device__ __forceinline__ void topk_gates_from(At at, int E, int k, int gating,
                                                int (&sel)[KMAX], float (&g)[KMAX]) {
    float val[KMAX];
#pragma unroll
    for (int p = 0; p < KMAX; ++p) {
        val[p] = -INFINITY;
        sel[p] = -1;
    }
    auto insert = [&](int e) {
        float v = at(e);
        int id = e;
#pragma unroll
        for (int p = 0; p < KMAX; ++p) {
            const bool gt = sel[p] < 0 || v > val[p] || (v == val[p] && id < sel[p]);
            const float tv = val[p];
            const int ti = sel[p];
            val[p] = gt ? v : tv;
            sel[p] = gt ? id : ti;
            v = gt ? tv : v;
            id = gt ? ti : id;
        }
    };
    if constexpr (EMAX > 0) {
#pragma unroll
        for (int e = 0; e < EMAX; ++e)
            if (e < E) insert(e);
    } else {
        for (int e = 0; e < E; ++e) insert(e);
    }
    float z[KMAX];
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        z[j] = 0.f;
        if (j < k) {
            z[j] = expf(val[j] - val[0]);
            s += z[j];
        }
    }
    if (gating == MOE_GATING_SOFTMAX_TOPK) {
        s = 0.f;
        if constexpr (EMAX > 0) {
#pragma unroll
            for (int e = 0; e < EMAX; ++e)
                if (e < E) s += expf(at(e) - val[0]);
        } else {
            for (int e = 0; e < E; ++e) s += expf(at(e) - val[0]);
        }
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j) g[j] = z[j] / s;
}

template <int KMAX>
__device__ __forceinline__ void topk_gates(const float *l, int E, int k, int gating,
                                           int (&sel)[KMAX], float (&g)[KMAX]) {
    topk_gates_from<KMAX, 0>([l](int e) { return l[e]; }, E, k, gating, sel, g);
}

}  // namespace moe
