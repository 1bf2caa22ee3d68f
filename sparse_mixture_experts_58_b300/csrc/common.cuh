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

// Selection of the k (<= 2) largest of E logits: slot 0 gets the largest,
// equal values go to the lower index.  Gates: softmax over the kept logits,
// computed relative to the largest so the exponent is <= 0.
__device__ __forceinline__ void top2_gates(const float *l, int E, int k, int *sel, float *g) {
    int i0 = 0;
    float b0 = l[0];
    int i1 = -1;
    float b1 = 0.f;
    for (int e = 1; e < E; ++e) {
        float v = l[e];
        if (v > b0) {
            i1 = i0; b1 = b0;
            i0 = e;  b0 = v;
        } else if (i1 < 0 || v > b1) {
            i1 = e;  b1 = v;
        }
    }
    sel[0] = i0;
    if (k == 1) {
        g[0] = 1.f;
        return;
    }
    sel[1] = i1;
    float z = expf(b1 - b0);
    float s = 1.f + z;
    g[0] = 1.f / s;
    g[1] = z / s;
}

}  // namespace moe
