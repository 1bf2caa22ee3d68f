// Grouped expert GEMMs in plain fp32 FMAs (never TF32), for fp32 layers.
// Same work decomposition as the tensor-core path -- units of (expert, tile
// of 64 rows, tile of 64 output columns) built from the device-side row
// offsets -- with a classic shared-memory-tiled SIMT inner loop.  Every
// output sums its contraction in index order.
#include "internal.h"

namespace moe {
namespace {

constexpr int kMaxE = MOE_MAX_EXPERTS;
constexpr int BM = 64, BN = 64, BK = 16;

struct SimtArgs {
    const float *B0[kMaxE];  // W1[e] or W2[e]: [N][K]
    const float *B1[kMaxE];  // W3[e] (SwiGLU only)
    const int *offsets;      // [E + 1]
    const float *A;          // [rows][K]
    float *out;              // [rows][N]
    int E, rows, K, N;
};

template <bool SWIGLU>
__global__ void __launch_bounds__(256) grouped_gemm_f32(const __grid_constant__ SimtArgs a) {
    __shared__ float sA[BK][BM + 4];
    __shared__ float sB0[BK][BN + 4];
    __shared__ float sB1[SWIGLU ? BK : 1][BN + 4];
    __shared__ int s_off[kMaxE + 1], s_mt[kMaxE], s_ustart[kMaxE + 1];

    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x;
    const int NT = (a.N + BN - 1) / BN;
    if (tid <= a.E) s_off[tid] = a.offsets[tid];
    __syncthreads();
    if (tid == 0) {
        int acc = 0;
        for (int e = 0; e < a.E; ++e) {
            const int cnt = s_off[e + 1] - s_off[e];
            s_mt[e] = (cnt + BM - 1) / BM;
            s_ustart[e] = acc;
            acc += s_mt[e] * NT;
        }
        s_ustart[a.E] = acc;
    }
    __syncthreads();
    const int u = blockIdx.x;
    if (u >= s_ustart[a.E]) return;
    int e = 0;
    while (e + 1 < a.E && u >= s_ustart[e + 1]) ++e;
    const int local = u - s_ustart[e];
    const int mt = local % s_mt[e];
    const int n0 = (local / s_mt[e]) * BN;
    const int row0 = s_off[e] + mt * BM;
    const int nrows = min(BM, s_off[e + 1] - row0);
    const float *B0 = a.B0[e];
    const float *B1 = SWIGLU ? a.B1[e] : nullptr;

    const int ty = tid / 16, tx = tid % 16;
    float acc0[4][4] = {}, acc1[4][4] = {};
    const int lrow = tid / 4, lk = (tid % 4) * 4;
    for (int k0 = 0; k0 < a.K; k0 += BK) {
        // token tile (transposed into shared memory)
        {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (lrow < nrows && k0 + lk < a.K)
                v = *reinterpret_cast<const float4 *>(a.A + (size_t)(row0 + lrow) * a.K + k0 + lk);
            sA[lk + 0][lrow] = v.x;
            sA[lk + 1][lrow] = v.y;
            sA[lk + 2][lrow] = v.z;
            sA[lk + 3][lrow] = v.w;
        }
        // weight tile(s)
        {
            const int n = n0 + lrow;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f), w = v;
            if (n < a.N && k0 + lk < a.K) {
                v = *reinterpret_cast<const float4 *>(B0 + (size_t)n * a.K + k0 + lk);
                if (SWIGLU) w = *reinterpret_cast<const float4 *>(B1 + (size_t)n * a.K + k0 + lk);
            }
            sB0[lk + 0][lrow] = v.x;
            sB0[lk + 1][lrow] = v.y;
            sB0[lk + 2][lrow] = v.z;
            sB0[lk + 3][lrow] = v.w;
            if (SWIGLU) {
                sB1[lk + 0][lrow] = w.x;
                sB1[lk + 1][lrow] = w.y;
                sB1[lk + 2][lrow] = w.z;
                sB1[lk + 3][lrow] = w.w;
            }
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float av[4], bv[4], cv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                av[i] = sA[kk][ty * 4 + i];
                bv[i] = sB0[kk][tx * 4 + i];
                if (SWIGLU) cv[i] = sB1[kk][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc0[i][j] = fmaf(av[i], bv[j], acc0[i][j]);
                    if (SWIGLU) acc1[i][j] = fmaf(av[i], cv[j], acc1[i][j]);
                }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = ty * 4 + i;
        if (r >= nrows) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= a.N) continue;
            float v = acc0[i][j];
            if (SWIGLU) v = v / (1.f + expf(-v)) * acc1[i][j];
            a.out[(size_t)(row0 + r) * a.N + n] = v;
        }
    }
}

template <bool SWIGLU>
cudaError_t run_f32(const float *A, const int *offsets, const void *const *B0,
                    const void *const *B1, int rows, int K, int N, int E, float *out,
                    cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    SimtArgs args;
    for (int e = 0; e < E; ++e) {
        args.B0[e] = static_cast<const float *>(B0[e]);
        args.B1[e] = SWIGLU ? static_cast<const float *>(B1[e]) : nullptr;
    }
    args.offsets = offsets;
    args.A = A;
    args.out = out;
    args.E = E;
    args.rows = rows;
    args.K = K;
    args.N = N;
    const int grid = ((rows + BM - 1) / BM + E) * ((N + BN - 1) / BN);
    return launch_pdl(grouped_gemm_f32<SWIGLU>, grid, 256, 0, s, args);
}

}  // namespace

cudaError_t launch_swiglu_f32(const float *x_perm, const int *offsets, const void *const *W1,
                              const void *const *W3, int rows, int d, int ffn, int E, float *h,
                              cudaStream_t s) {
    return run_f32<true>(x_perm, offsets, W1, W3, rows, d, ffn, E, h, s);
}

cudaError_t launch_down_f32(const float *h, const int *offsets, const void *const *W2, int rows,
                            int d, int ffn, int E, float *y, cudaStream_t s) {
    return run_f32<false>(h, offsets, W2, nullptr, rows, ffn, d, E, y, s);
}

}  // namespace moe
