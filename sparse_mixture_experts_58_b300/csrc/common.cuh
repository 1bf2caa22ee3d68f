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

// Selection of the k (<= MOE_MAX_TOPK) largest of E logits by insertion into
// a descending list: slot 0 gets the largest; a value only moves ahead of a
// strictly smaller one, so equal values keep ascending expert order.
// Gates, relative to the largest logit l0 so every exponent is <= 0:
//   gating 0: z_j = exp(l_j - l0), g_j = z_j / sum_j' z_j' (softmax over kept);
//   gating 1: g_j = exp(l_j - l0) / sum_e exp(l_e - l0) (full softmax, kept
//             entries not renormalised).
__device__ __forceinline__ void topk_gates(const float *l, int E, int k, int gating, int *sel,
                                           float *g) {
    float val[MOE_MAX_TOPK];
    int n = 0;
    for (int e = 0; e < E; ++e) {
        const float v = l[e];
        if (n < k || v > val[n - 1]) {
            int p = n < k ? n : k - 1;
            while (p > 0 && v > val[p - 1]) {
                val[p] = val[p - 1];
                sel[p] = sel[p - 1];
                --p;
            }
            val[p] = v;
            sel[p] = e;
            if (n < k) ++n;
        }
    }
    float z[MOE_MAX_TOPK];
    float s = 0.f;
    for (int j = 0; j < k; ++j) {
        z[j] = expf(val[j] - val[0]);
        s += z[j];
    }
    if (gating == MOE_GATING_SOFTMAX_TOPK) {
        s = 0.f;
        for (int e = 0; e < E; ++e) s += expf(l[e] - val[0]);
    }
    for (int j = 0; j < k; ++j) g[j] = z[j] / s;
}

}  // namespace moe
