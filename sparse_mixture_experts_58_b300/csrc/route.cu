// Grouping tokens by expert: the chosen experts' rows are laid out expert by
// expert, tokens ascending inside each expert, so every expert's input is one
// contiguous block of rows ("Mixtral" curriculum page: run only the chosen
// MLPs; batching tokens per expert is the routing work of MoE serving).
//
//   chunk_scan:   per-expert exclusive scan over the router's per-chunk counts
//                 -> counts[E], offsets[E+1], chunk_base[chunk][E]
//   group_tokens: row of (t, j) = offsets[e] + chunk_base[chunk][e] + rank of
//                 t among the chunk's tokens routed to e; writes perm / inv and
//                 copies x[t] to each of its rows (16-byte vectors).
// No atomics decide any position, so the result is deterministic.
#include "internal.h"

namespace moe {
namespace {

// One block of 1024 threads; warp e scans expert e's column of chunk counts.
__global__ void __launch_bounds__(1024) chunk_scan_kernel(const int *__restrict__ cc, int nchunks,
                                                          int E, int *chunk_base, int *counts,
                                                          int *offsets) {
    __shared__ int s_tot[MOE_MAX_EXPERTS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < E) {
        int carry = 0;
        for (int base = 0; base < nchunks; base += 32) {
            const int c = base + lane;
            const int v = c < nchunks ? cc[(size_t)c * E + warp] : 0;
            int s = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, s, off);
                if (lane >= off) s += n;
            }
            if (c < nchunks) chunk_base[(size_t)c * E + warp] = carry + s - v;
            carry += __shfl_sync(0xffffffffu, s, 31);
        }
        if (lane == 0) s_tot[warp] = carry;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        offsets[0] = 0;
        for (int e = 0; e < E; ++e) {
            counts[e] = s_tot[e];
            acc += s_tot[e];
            offsets[e + 1] = acc;
        }
    }
}

// Copy one row (rowvec 16-byte vectors) from src to k destinations.
__device__ __forceinline__ void copy_row(const uint4 *__restrict__ src, uint4 *dst0, uint4 *dst1,
                                         int rowvec, int lane) {
#pragma unroll 4
    for (int v = lane; v < rowvec; v += 32) {
        const uint4 val = __ldcs(src + v);
        dst0[v] = val;
        if (dst1 != nullptr) dst1[v] = val;
    }
}

// One block = one chunk of kChunk tokens (8 warps x 2 tokens for the copy).
__global__ void __launch_bounds__(256) group_tokens_kernel(
    const int *__restrict__ idx, const int *__restrict__ chunk_base,
    const int *__restrict__ offsets, const uint8_t *__restrict__ x, int Tn, int E, int k,
    size_t row_bytes, int *perm, int *inv, uint8_t *x_perm) {
    __shared__ int s_idx[kChunk * 2];
    __shared__ int s_row[kChunk * 2];
    const int c = blockIdx.x;
    const int first = c * kChunk;
    const int ntok = min(kChunk, Tn - first);
    if (threadIdx.x < ntok * k) s_idx[threadIdx.x] = idx[(size_t)first * k + threadIdx.x];
    __syncthreads();
    if (threadIdx.x < ntok) {
        const int i = threadIdx.x;
        const int t = first + i;
        for (int j = 0; j < k; ++j) {
            const int e = s_idx[i * k + j];
            int rank = 0;
            for (int i2 = 0; i2 < i; ++i2)
                for (int j2 = 0; j2 < k; ++j2) rank += (s_idx[i2 * k + j2] == e);
            const int r = offsets[e] + chunk_base[(size_t)c * E + e] + rank;
            perm[r] = t * k + j;
            inv[(size_t)t * k + j] = r;
            s_row[i * k + j] = r;
        }
    }
    if (x == nullptr) return;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rowvec = static_cast<int>(row_bytes / 16);
    for (int i = warp * 2; i < warp * 2 + 2 && i < ntok; ++i) {
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)(first + i) * row_bytes);
        uint4 *d0 = reinterpret_cast<uint4 *>(x_perm + (size_t)s_row[i * k] * row_bytes);
        uint4 *d1 = k > 1 ? reinterpret_cast<uint4 *>(x_perm + (size_t)s_row[i * k + 1] * row_bytes)
                          : nullptr;
        copy_row(src, d0, d1, rowvec, lane);
    }
}

// x_perm[r] = x[perm[r] / k]: one warp per row.
__global__ void __launch_bounds__(256) permute_kernel(const uint8_t *__restrict__ x,
                                                      const int *__restrict__ perm, int rows, int k,
                                                      size_t row_bytes, uint8_t *x_perm) {
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= rows) return;
    const int t = perm[r] / k;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * row_bytes);
    uint4 *dst = reinterpret_cast<uint4 *>(x_perm + (size_t)r * row_bytes);
    copy_row(src, dst, nullptr, static_cast<int>(row_bytes / 16), threadIdx.x & 31);
}

}  // namespace

cudaError_t launch_chunk_scan(const int *chunk_counts, int nchunks, int E, int *chunk_base,
                              int *counts, int *offsets, cudaStream_t s) {
    chunk_scan_kernel<<<1, 1024, 0, s>>>(chunk_counts, nchunks, E, chunk_base, counts, offsets);
    return cudaGetLastError();
}

cudaError_t launch_group_tokens(const int *idx, const int *chunk_base, const int *offsets,
                                const void *x, int T, int d, int E, int k, int elt, int *perm,
                                int *inv, void *x_perm, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int nchunks = (T + kChunk - 1) / kChunk;
    group_tokens_kernel<<<nchunks, 256, 0, s>>>(
        idx, chunk_base, offsets, static_cast<const uint8_t *>(x), T, E, k, (size_t)d * elt, perm,
        inv, static_cast<uint8_t *>(x_perm));
    return cudaGetLastError();
}

cudaError_t launch_permute(const void *x, const int *perm, int T, int d, int k, int elt,
                           void *x_perm, cudaStream_t s) {
    const int rows = T * k;
    if (rows == 0) return cudaSuccess;
    permute_kernel<<<(rows + 7) / 8, 256, 0, s>>>(static_cast<const uint8_t *>(x), perm, rows, k,
                                                  (size_t)d * elt, static_cast<uint8_t *>(x_perm));
    return cudaGetLastError();
}

}  // namespace moe
