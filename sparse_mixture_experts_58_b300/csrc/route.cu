// Grouping tokens by expert: the chosen experts' rows are laid out expert by
// expert, tokens ascending inside each expert, so every expert's input is one
// contiguous block of rows ("Mixtral" curriculum page: run only the chosen
// MLPs; batching tokens per expert is the routing work of MoE serving).
//
//   chunk_scan:   per chunk of kChunk tokens, how many selections hit each
//                 expert; per expert, the exclusive scan of those counts over
//                 chunks (a selection's rank among its expert's selections in
//                 token order = chunk base + rank inside the chunk); counts and
//                 offsets of the rows each expert keeps (all of them, or the
//                 first `capacity` in token order).
//   group_tokens: row of (t, j) = offsets[e] + rank, or dropped when rank >=
//                 capacity; writes perm / inv and copies x[t] to each of its
//                 rows (16-byte vectors).
// No atomics decide any position, so the result is deterministic.
#include "internal.h"

namespace moe {
namespace {

// One block of 1024 threads.  First each warp counts, for its chunks, how many
// of the chunk's kChunk*k selections hit each expert (ballots over 32-lane
// segments of idx); lane e%32 keeps expert e's count.  The counts go through
// global memory (cc); __syncthreads() orders the block's writes before its
// reads.  Then warp w scans the columns of experts w and w + 32.
__global__ void __launch_bounds__(1024) chunk_scan_kernel(const int *__restrict__ idx, int Tn,
                                                          int k, int E, int capacity, int pad,
                                                          int *cc, int *chunk_base, int *counts,
                                                          int *offsets) {
    __shared__ int s_tot[MOE_MAX_EXPERTS];
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nchunks = (Tn + kChunk - 1) / kChunk;
    for (int c = warp; c < nchunks; c += 32) {
        const int first = c * kChunk;
        const int nsel = min(kChunk, Tn - first) * k;
        int mine_lo = 0, mine_hi = 0;  // experts lane and lane + 32
        for (int s0 = 0; s0 < nsel; s0 += 32) {
            const int sel = s0 + lane < nsel ? idx[(size_t)first * k + s0 + lane] : -1;
            for (int e = 0; e < E; ++e) {
                const int n = __popc(__ballot_sync(0xffffffffu, sel == e));
                if (lane == e) mine_lo += n;
                if (lane + 32 == e) mine_hi += n;
            }
        }
        if (lane < E) cc[(size_t)c * E + lane] = mine_lo;
        if (lane + 32 < E) cc[(size_t)c * E + lane + 32] = mine_hi;
    }
    __syncthreads();
    for (int e = warp; e < E; e += 32) {
        int carry = 0;
        for (int base = 0; base < nchunks; base += 32) {
            const int c = base + lane;
            const int v = c < nchunks ? cc[(size_t)c * E + e] : 0;
            int s = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, s, off);
                if (lane >= off) s += n;
            }
            if (c < nchunks) chunk_base[(size_t)c * E + e] = carry + s - v;
            carry += __shfl_sync(0xffffffffu, s, 31);
        }
        if (lane == 0) s_tot[e] = capacity > 0 ? min(carry, capacity) : carry;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        offsets[0] = 0;
        for (int e = 0; e < E; ++e) {
            counts[e] = s_tot[e];
            acc += (s_tot[e] + pad - 1) / pad * pad;
            offsets[e + 1] = acc;
        }
    }
}

// The whole grouping of a small batch (n = T * k <= kRouteSmallMax
// selections) in one block: counts, offsets, perm, inv and the row copies,
// in place of chunk_scan + group_tokens.  Selections are taken in order
// s = t * k + j, in chunks of 32 (one per warp at a time).  Per chunk, the
// lanes that hold the same expert find each other (match), the lowest of them
// records the chunk's count for that expert; a scan over chunks per expert
// gives each chunk's base; a selection's rank is its chunk's base plus the
// matching lanes below it, so the row order is (expert, token) as in the two
// kernels, and the results are the same.  Then the kept rows are copied
// (row_scale: scaled and rounded, the fused RMSNorm), the copy split evenly
// over the grid's blocks; every block ranks the (few) selections itself and
// block 0 alone writes counts, offsets, perm and inv.
constexpr int kRouteSmallMax = 1024;
constexpr int kRouteSmallChunks = kRouteSmallMax / 32;

template <typename T>
__global__ void __launch_bounds__(1024) route_small_kernel(
    const int *__restrict__ idx, int n, int k, int E, int capacity, const T *__restrict__ x,
    const float *__restrict__ row_scale, int d, int *counts, int *offsets, int *perm, int *inv,
    T *x_perm, int *zero_ctr, int nzero) {
    __shared__ int s_sel[kRouteSmallMax];
    __shared__ int s_src[kRouteSmallMax];  // row -> source token
    __shared__ uint8_t s_cnt[kRouteSmallChunks][MOE_MAX_EXPERTS];
    __shared__ uint16_t s_base[kRouteSmallChunks][MOE_MAX_EXPERTS];
    __shared__ int s_tot[MOE_MAX_EXPERTS];
    __shared__ int s_off[MOE_MAX_EXPERTS + 1];
    pdl_wait();
    pdl_trigger();
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero_ctr[i] = 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int nch = (n + 31) / 32;
    for (int i = threadIdx.x; i < nch * MOE_MAX_EXPERTS; i += blockDim.x)
        s_cnt[i / MOE_MAX_EXPERTS][i % MOE_MAX_EXPERTS] = 0;
    __syncthreads();
    for (int c = warp; c < nch; c += nwarps) {
        const int s0 = 32 * c + lane;
        const int sel = s0 < n ? idx[s0] : -1;
        s_sel[s0] = sel;
        const unsigned m = __match_any_sync(0xffffffffu, sel);
        if (sel >= 0 && (m & ((1u << lane) - 1u)) == 0) s_cnt[c][sel] = (uint8_t)__popc(m);
    }
    __syncthreads();
    for (int e = warp; e < E; e += nwarps) {
        int carry = 0;
        for (int base = 0; base < nch; base += 32) {
            const int c = base + lane;
            const int v = c < nch ? s_cnt[c][e] : 0;
            int sc = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, sc, off);
                if (lane >= off) sc += t;
            }
            if (c < nch) s_base[c][e] = (uint16_t)(carry + sc - v);
            carry += __shfl_sync(0xffffffffu, sc, 31);
        }
        if (lane == 0) s_tot[e] = capacity > 0 ? min(carry, capacity) : carry;
    }
    __syncthreads();
    const bool writer = blockIdx.x == 0;
    if (threadIdx.x == 0) {
        int acc = 0;
        s_off[0] = 0;
        for (int e = 0; e < E; ++e) {
            if (writer) counts[e] = s_tot[e];
            acc += s_tot[e];
            s_off[e + 1] = acc;
        }
    }
    __syncthreads();
    if (writer)
        for (int i = threadIdx.x; i <= E; i += blockDim.x) offsets[i] = s_off[i];
    for (int c = warp; c < nch; c += nwarps) {
        const int s0 = 32 * c + lane;
        const int sel = s_sel[s0];
        const unsigned m = __match_any_sync(0xffffffffu, sel);
        if (sel >= 0) {
            const int rank = s_base[c][sel] + __popc(m & ((1u << lane) - 1u));
            const bool kept = capacity <= 0 || rank < capacity;
            const int r = kept ? s_off[sel] + rank : -1;
            if (writer) inv[s0] = r;
            if (kept) {
                if (writer) perm[r] = s0;
                s_src[r] = s0 / k;
            }
        }
    }
    __syncthreads();
    // rows r < offsets[E]: x_perm[r] = x[source token], flattened to (row,
    // 16-byte vector); this block's share of them, U loads in flight per thread
    constexpr int VN = Vec<T>::n;
    constexpr int U = 8;
    const int rowvec = d / VN;
    const int all = s_off[E] * rowvec;
    const int beg = (int)((long long)all * blockIdx.x / gridDim.x);
    const int total = (int)((long long)all * (blockIdx.x + 1) / gridDim.x);
    for (int i0 = beg + threadIdx.x; i0 < total; i0 += blockDim.x * U) {
        uint4 val[U];
        int row[U], vec[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + blockDim.x * u;
            const int ii = i < total ? i : beg;
            row[u] = ii / rowvec;
            vec[u] = ii - row[u] * rowvec;
            val[u] = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)s_src[row[u]] * d) + vec[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (i0 + (int)blockDim.x * u < total) {
                const uint4 v = row_scale != nullptr
                                    ? scale_slice<T>(val[u], row_scale[s_src[row[u]]])
                                    : val[u];
                reinterpret_cast<uint4 *>(x_perm + (size_t)row[u] * d)[vec[u]] = v;
            }
        }
    }
}

// Copy one row (rowvec 16-byte vectors) from src to one destination, one
// warp; four loads per lane are issued before their stores.
__device__ __forceinline__ void copy_row(const uint4 *__restrict__ src, uint4 *dst, int rowvec,
                                         int lane) {
    constexpr int U = 4;
    for (int v0 = lane; v0 < rowvec; v0 += 32 * U) {
        uint4 val[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + 32 * u;
            val[u] = __ldcs(src + (v < rowvec ? v : 0));
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + 32 * u;
            if (v < rowvec) dst[v] = val[u];
        }
    }
}

// One block = one chunk of kChunk tokens (x up to 8 row slices for small
// batches, blockIdx.y).  Thread i < kChunk ranks token i's selections against
// the chunk's earlier tokens; then all threads copy rows.  With row_scale
// (elt 2: bf16, 4: fp32), each 16-byte slice is multiplied by its token's
// scale and rounded to the storage type on the way.
template <int KMAX>
__global__ void __launch_bounds__(256) group_tokens_kernel(
    const int *__restrict__ idx, const int *__restrict__ chunk_base,
    const int *__restrict__ offsets, const uint8_t *__restrict__ x,
    const float *__restrict__ row_scale, int elt, int Tn, int E, int k, int capacity,
    size_t row_bytes, int *perm, int *inv, uint8_t *x_perm, float *zero_acc) {
    __shared__ int s_idx[kChunk * MOE_MAX_TOPK];
    __shared__ int s_row[kChunk * MOE_MAX_TOPK];
    __shared__ float s_scale[kChunk];
    pdl_wait();
    pdl_trigger();
    const int c = blockIdx.x;
    const int first = c * kChunk;
    const int ntok = min(kChunk, Tn - first);
    for (int i = threadIdx.x; i < ntok * k; i += blockDim.x)
        s_idx[i] = idx[(size_t)first * k + i];
    if (row_scale != nullptr && threadIdx.x < ntok)
        s_scale[threadIdx.x] = row_scale[first + threadIdx.x];
    __syncthreads();
    if (threadIdx.x < ntok) {
        const int i = threadIdx.x;
        const int t = first + i;
        for (int j = 0; j < k; ++j) {
            const int e = s_idx[i * k + j];
            int rank = 0;
            for (int i2 = 0; i2 < i; ++i2)
                for (int j2 = 0; j2 < k; ++j2) rank += (s_idx[i2 * k + j2] == e);
            rank += chunk_base[(size_t)c * E + e];
            const bool kept = capacity <= 0 || rank < capacity;
            const int r = kept ? offsets[e] + rank : -1;
            if (blockIdx.y == 0) {
                if (kept) perm[r] = t * k + j;
                inv[(size_t)t * k + j] = r;
            }
            s_row[i * k + j] = r;
        }
    }
    if (x == nullptr) return;
    __syncthreads();
    // This block's slice of the chunk's rows (blockIdx.y of gridDim.y parts),
    // flattened to (token, 16-byte vector) pairs over all threads; each thread
    // issues U loads, then writes each value to the token's kept rows.
    constexpr int U = 8;
    const int rowvec_all = static_cast<int>(row_bytes / 16);
    const int vbeg = (int)((long long)rowvec_all * blockIdx.y / gridDim.y);
    const int vend = (int)((long long)rowvec_all * (blockIdx.y + 1) / gridDim.y);
    if (zero_acc != nullptr) {
        // the same columns of the tokens' fp32 accumulator rows (4 / elt
        // float4 per 16-byte vector of x)
        const int per = 4 / elt;
        const int nf4 = (vend - vbeg) * per, f4_all = rowvec_all * per;
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        float4 *acc4 = reinterpret_cast<float4 *>(zero_acc) + (size_t)first * f4_all + vbeg * per;
        for (int i = threadIdx.x; i < ntok * nf4; i += blockDim.x) {
            const int tk = i / nf4;
            acc4[(size_t)tk * f4_all + (i - tk * nf4)] = z;
        }
    }
    const int rowvec = vend - vbeg;
    const int total = ntok * rowvec;
    const uint4 *xs = reinterpret_cast<const uint4 *>(x + (size_t)first * row_bytes);
    for (int i0 = threadIdx.x; i0 < total; i0 += blockDim.x * U) {
        uint4 val[U];
        int tok[U], vec[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + blockDim.x * u;
            const int ii = i < total ? i : 0;
            tok[u] = ii / rowvec;
            vec[u] = vbeg + (ii - tok[u] * rowvec);
            val[u] = __ldcs(xs + (size_t)tok[u] * rowvec_all + vec[u]);
        }
        if (row_scale != nullptr) {
#pragma unroll
            for (int u = 0; u < U; ++u)
                val[u] = elt == 2 ? scale_slice<__nv_bfloat16>(val[u], s_scale[tok[u]])
                                  : scale_slice<float>(val[u], s_scale[tok[u]]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (i0 + (int)blockDim.x * u < total) {
#pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    if (j < k) {
                        const int r = s_row[tok[u] * k + j];
                        if (r >= 0)
                            reinterpret_cast<uint4 *>(x_perm + (size_t)r * row_bytes)[vec[u]] =
                                val[u];
                    }
                }
            }
        }
    }
}

// x_perm[r] = x[perm[r] / k]: one warp per row.
__global__ void __launch_bounds__(256) permute_kernel(const uint8_t *__restrict__ x,
                                                      const int *__restrict__ perm, int rows, int k,
                                                      size_t row_bytes, uint8_t *x_perm) {
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= rows) return;
    const int t = perm[r] / k;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * row_bytes);
    uint4 *dst = reinterpret_cast<uint4 *>(x_perm + (size_t)r * row_bytes);
    copy_row(src, dst, static_cast<int>(row_bytes / 16), threadIdx.x & 31);
}

}  // namespace

cudaError_t launch_chunk_scan(const int *idx, int T, int k, int E, int capacity, int *chunk_counts,
                              int *chunk_base, int *counts, int *offsets, cudaStream_t s, int pad) {
    return launch_pdl(chunk_scan_kernel, 1, 1024, 0, s, idx, T, k, E, capacity, pad, chunk_counts,
                      chunk_base, counts, offsets);
}

cudaError_t launch_group_tokens(const int *idx, const int *chunk_base, const int *offsets,
                                const void *x, const float *row_scale, int T, int d, int E, int k,
                                int capacity, int elt, int *perm, int *inv, void *x_perm,
                                cudaStream_t s, float *zero_acc) {
    if (T == 0) return cudaSuccess;
    const int nchunks = (T + kChunk - 1) / kChunk;
    // few chunks (small batches): split each chunk's row copy over several
    // blocks so enough loads are in flight
    int parts = 1;
    if (x != nullptr) {
        const int rowvec = (int)((size_t)d * elt / 16);
        parts = (2 * kPlanSms + nchunks - 1) / nchunks;
        if (parts > 8) parts = 8;
        if (parts > rowvec) parts = rowvec > 0 ? rowvec : 1;
        if (parts < 1) parts = 1;
    }
    if (k <= 2)
        return launch_pdl(group_tokens_kernel<2>, dim3(nchunks, parts), 256, 0, s, idx,
                          chunk_base, offsets, static_cast<const uint8_t *>(x), row_scale, elt, T,
                          E, k, capacity, (size_t)d * elt, perm, inv,
                          static_cast<uint8_t *>(x_perm), zero_acc);
    return launch_pdl(group_tokens_kernel<MOE_MAX_TOPK>, dim3(nchunks, parts), 256, 0, s, idx,
                      chunk_base, offsets, static_cast<const uint8_t *>(x), row_scale, elt, T, E,
                      k, capacity, (size_t)d * elt, perm, inv, static_cast<uint8_t *>(x_perm),
                      zero_acc);
}

int route_small_max() { return kRouteSmallMax; }

cudaError_t launch_route_small(const int *idx, int T, int k, int E, int capacity, const void *x,
                               const float *row_scale, int d, int elt, int *counts, int *offsets,
                               int *perm, int *inv, void *x_perm, cudaStream_t s, int *zero_ctr,
                               int nzero) {
    const int n = T * k;
    if (n > kRouteSmallMax || E > MOE_MAX_EXPERTS) return cudaErrorInvalidValue;
    // a warp per 32-selection chunk (at least 4, at most 32); one block per
    // 16 KB of rows to copy, at most 32 (each ranks the selections itself)
    int warps = (n + 31) / 32;
    if (warps < 4) warps = 4;
    if (warps > 32) warps = 32;
    const long long copy_bytes = (long long)n * d * elt;
    int blocks = (int)((copy_bytes + (16 << 10) - 1) / (16 << 10));
    if (blocks < 1) blocks = 1;
    if (blocks > 32) blocks = 32;
    const int threads = warps < 8 ? 256 : 32 * warps;
    if (elt == 2)
        return launch_pdl(route_small_kernel<__nv_bfloat16>, blocks, threads, 0, s, idx, n, k,
                          E, capacity, static_cast<const __nv_bfloat16 *>(x), row_scale, d,
                          counts, offsets, perm, inv, static_cast<__nv_bfloat16 *>(x_perm),
                          zero_ctr, nzero);
    return launch_pdl(route_small_kernel<float>, blocks, threads, 0, s, idx, n, k, E, capacity,
                      static_cast<const float *>(x), row_scale, d, counts, offsets, perm, inv,
                      static_cast<float *>(x_perm), zero_ctr, nzero);
}

cudaError_t launch_permute(const void *x, const int *perm, int rows, int d, int k, int elt,
                           void *x_perm, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    return launch_pdl(permute_kernel, (rows + 7) / 8, 256, 0, s, static_cast<const uint8_t *>(x),
                      perm, rows, k, (size_t)d * elt, static_cast<uint8_t *>(x_perm));
}

}  // namespace moe
