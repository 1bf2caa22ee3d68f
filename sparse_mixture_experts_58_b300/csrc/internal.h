// Host-side declarations shared by the libmoe translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include "common.cuh"

namespace moe {

// SM count the tile planner sizes work for (a B300 has 148); grids use the
// device's real count at launch.
constexpr int kPlanSms = 148;

// How one call is carved into kernels and scratch.
struct Plan {
    int T, d, ffn, E, k, dt;
    int rows;      // T * k expert rows
    int nchunks;   // router chunks of kChunk tokens
    // grouped expert GEMMs (bf16 tensor-core path)
    int wide;      // 1: 256-wide tiles (many rows per expert); 0: 128-wide
    int pair;      // 1: CTA pairs, 256 weight rows x up to 256 token rows per tile
    int bm;        // token rows per tile (<= 128)
    int splits;    // split of the down projection's contraction
    int kps;       // 64-wide contraction blocks per split
    int small_route;  // 1: one kernel groups the batch (scan, ranks, row copies)
    int fuse;      // 1: the down projection's epilogue adds gate x output into
                   // a zeroed fp32 row per token (the combine), a finalize
                   // pass rounds it; needs k <= 2, one split, the pair kernel
    int gsplit;    // 1: the gate/up GEMM may split its contraction in two (the
                   // kernel decides from the busy experts); counters zeroed by
                   // the one-kernel grouping
    int nctr;      // gate/up split arrival counters
    // workspace layout (byte offsets, 256-aligned)
    size_t o_logits, o_idx, o_gates, o_ccount, o_cbase, o_counts, o_offsets, o_perm, o_inv;
    size_t o_rms;  // per-token RMSNorm scale (pre-norm blocks)
    size_t o_xperm, o_h, o_y, o_gpart, o_gctr, bytes;
};

int make_plan(int T, int d, int ffn, int E, int k, int dt, Plan *p);

// moe_forward's validation and launch sequence, enqueued directly on the
// stream (no launch graph); the library's fixed-scratch entry point uses it.
int forward_direct(const void *x, const void *W_g, const float *router_bias,
                   const void *const *W1, const void *const *W3, const void *const *W2, int T,
                   int d, int ffn, int E, int k, int dtype, void *out, void *workspace,
                   size_t workspace_bytes, cudaStream_t s);

// Launch with programmatic stream serialisation allowed, so the kernel may be
// scheduled while the previous kernel on the stream drains (the kernel itself
// calls pdl_wait() before reading earlier results).  A previous kernel that
// never triggers releases it at completion, as an ordinary launch would.
// Whether launches carry the attribute (MOE_PDL=1; off by default).
bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

int elem_size(int dt);
int device_sm_count();
// Device address of the status word for the current device (nullptr on error).
int *device_status_ptr();

// Kernel launchers (each returns the launch's cudaError_t).
// inv_rms != nullptr: RMSNorm (eps) fused in front of the router; each
// token's scale is written to inv_rms[T].
// x_copy != nullptr: x is page-locked host memory (the device's address of
// it) read over the bus, and the router also copies the rows to x_copy in
// device memory; only where router_reads_host_rows(T, E) (one pass over the
// rows, no fused RMSNorm).
cudaError_t launch_router(const void *x, const void *Wg, const float *bias, int T, int d, int E,
                          int k, int dt, int gating, float eps, float *inv_rms, float *logits,
                          int *idx, float *gates, cudaStream_t s, void *x_copy = nullptr);
bool router_reads_host_rows(int T, int E);
cudaError_t launch_topk_from_logits(const float *logits, int T, int E, int k, int gating,
                                    int *idx, float *gates, cudaStream_t s);
// Per-chunk expert counts from idx (into chunk_counts), then their per-expert
// exclusive scan: chunk_base; counts and offsets of the kept rows (capacity
// <= 0: all rows).  pad > 1: each expert's block of rows starts on a multiple
// of pad (offsets[e + 1] - offsets[e] = counts[e] rounded up to pad).
cudaError_t launch_chunk_scan(const int *idx, int T, int k, int E, int capacity, int *chunk_counts,
                              int *chunk_base, int *counts, int *offsets, cudaStream_t s,
                              int pad = 1);
// row_scale != nullptr: each copied row is multiplied by its token's scale
// and rounded to the storage type (the fused RMSNorm).  zero_acc != nullptr: the chunk's
// rows of the fp32 [T][d] accumulator are set to zero.
cudaError_t launch_group_tokens(const int *idx, const int *chunk_base, const int *offsets,
                                const void *x, const float *row_scale, int T, int d, int E, int k,
                                int capacity, int elt, int *perm, int *inv, void *x_perm,
                                cudaStream_t s, float *zero_acc = nullptr);
// The grouping of a batch of at most route_small_max() selections (T * k) in
// one kernel: counts, offsets, perm, inv and the row copies (row_scale: the
// fused RMSNorm), as chunk_scan + group_tokens give them.  Block 0 also sets
// zero_ctr[0 .. nzero) to zero (the gate/up split's arrival counters).
int route_small_max();
cudaError_t launch_route_small(const int *idx, int T, int k, int E, int capacity, const void *x,
                               const float *row_scale, int d, int elt, int *counts, int *offsets,
                               int *perm, int *inv, void *x_perm, cudaStream_t s,
                               int *zero_ctr = nullptr, int nzero = 0);
// x_perm[r] = x[perm[r] / k] for r < rows.
cudaError_t launch_permute(const void *x, const int *perm, int rows, int d, int k, int elt,
                           void *x_perm, cudaStream_t s);

// Grouped expert GEMMs.  `rows` = total expert rows (T*k); `bm` rows per tile.
// gpart/gctr (both or neither; one-CTA kernel only): scratch for splitting the
// gate/up contraction in two where that shortens the rounds of units -- fp32
// partial sums [2][rows][2 ffn] and (rows / bm + E) * ceil(ffn / 56) arrival
// counters that must be zero at launch.
int launch_swiglu_tc(const void *x_perm, const int *offsets, const void *const *W1,
                     const void *const *W3, int rows, int d, int ffn, int E, int bm, int wide,
                     void *h, cudaStream_t s, float *gpart = nullptr, int *gctr = nullptr);
int launch_down_tc(const void *h, const int *offsets, const void *const *W2, int rows, int d,
                   int ffn, int E, int bm, int wide, int splits, int kps, float *y,
                   cudaStream_t s);
// The same on CTA pairs: 256 weight rows x up to 256 tokens (rounded to 16) per tile.
int launch_swiglu_pair(const void *x_perm, const int *offsets, const void *const *W1,
                       const void *const *W3, int rows, int d, int ffn, int E, void *h,
                       cudaStream_t s);
int launch_down_pair(const void *h, const int *offsets, const void *const *W2, int rows, int d,
                     int ffn, int E, int splits, int kps, float *y, cudaStream_t s);
// The down projection with the combine in its epilogue: for row r (token
// perm[r] / k, slot perm[r] % k) it adds gates[perm[r]] * y[r] into acc[token]
// (fp32 [T][d], zeroed beforehand); one split, k <= 2, so each element gets at
// most two additions into zero and the sum does not depend on their order.
int launch_down_pair_combine(const void *h, const int *offsets, const void *const *W2, int rows,
                             int d, int ffn, int E, const int *perm, const float *gates, int k,
                             float *acc, cudaStream_t s);
size_t pair_gemm_smem_bytes();

// Backward of the expert GEMMs (gemm_bwd.cu), on rows grouped by expert with
// each expert's block padded to a multiple of 64 (offsets).  rows: the row
// capacity of the row buffers.
int launch_bwd_uv(const void *x_rows, const int *offsets, const void *const *W1,
                  const void *const *W3, int rows, int d, int ffn, int E, void *U, void *V,
                  cudaStream_t s);
int launch_bwd_z(const void *g_rows, const int *offsets, const void *const *W2, int rows, int d,
                 int ffn, int E, const void *U, const void *V, const float *row_gate, void *dU,
                 void *dV, void *gH, float *dgp, cudaStream_t s);
int launch_bwd_dx(const void *dU, const void *dV, const int *offsets, const void *const *W1,
                  const void *const *W3, int rows, int d, int ffn, int E, float *dx_rows,
                  cudaStream_t s);
int launch_bwd_wgrad(const void *x_rows, const void *g_rows, const void *dU, const void *dV,
                     const void *gH, const int *offsets, int rows, int d, int ffn, int E,
                     float *const *dW1, float *const *dW3, float *const *dW2, cudaStream_t s);
size_t bwd_gemm_smem_bytes();

// Backward helpers (bwd.cu).  Rows r < offsets[E] of dst get src[perm[r] / k]
// (zero for padding rows, perm < 0); with gates, row_gate[r] = gates[perm[r]]
// (0 for padding).
cudaError_t launch_gather_rows(const void *src, const int *perm, const int *offsets, int E,
                               int rows, int k, int d, const float *gates, float *row_gate,
                               void *dst, cudaStream_t s);
// Per token: dg of each slot (sum of the dgp blocks of its row), the logit
// gradients of the kept softmax (dl [T][k]) and dx = sum_j dx_rows[row_j] +
// sum_j dl_j W_g[e_j], rounded once to bf16.
cudaError_t launch_router_bwd(const int *idx, const float *gates, const int *inv,
                              const float *dgp, int nblk, const float *dx_rows, const void *Wg,
                              int T, int d, int k, float *dl, void *dx, cudaStream_t s);
// dWg[e] = sum over tokens (in token order) of dl[t][j] x[t] for idx[t][j] = e;
// part: scratch of router_wg_part_floats(T, E, d) floats.
size_t router_wg_part_floats(int T, int E, int d);
cudaError_t launch_router_wgrad(const int *idx, const float *dl, const void *x, int T, int d,
                                int E, int k, float *part, float *dWg, cudaStream_t s);
cudaError_t launch_swiglu_f32(const float *x_perm, const int *offsets, const void *const *W1,
                              const void *const *W3, int rows, int d, int ffn, int E, float *h,
                              cudaStream_t s);
cudaError_t launch_down_f32(const float *h, const int *offsets, const void *const *W2, int rows,
                            int d, int ffn, int E, float *y, cudaStream_t s);

// residual != 0: out <- round(out + round(combined)) in place (the residual
// add of a pre-norm block).
cudaError_t launch_combine(const float *y, int splits, int rows, const float *gates,
                           const int *inv, int T, int d, int k, int renorm, int residual, int dt,
                           void *out, cudaStream_t s);
// out[t] = round(acc[t]) (residual != 0: out[t] <- round(out[t] + round(acc[t])))
// for the gated sums the down projection's epilogue accumulated.
cudaError_t launch_finalize(const float *acc, int T, int d, int residual, int dt, void *out,
                            cudaStream_t s);
cudaError_t launch_add_rmsnorm(void *x, const void *add, void *xn, int T, int d, float eps,
                               int dt, cudaStream_t s);
cudaError_t launch_wait_selftest(unsigned int limit_ns, cudaStream_t s);

// Tensor maps (TMA descriptors), encoded through the driver entry point.
int encode_map_bf16_2d(CUtensorMap *map, const void *base, unsigned long long inner,
                       unsigned long long outer, unsigned int box_inner,
                       unsigned int box_outer);
// W1[e] and W3[e] as one 4-D tensor whose box {64, 16, 2, 4} interleaves them
// in 16-row groups (see api.cu); MOE_ERR_UNSUPPORTED if the driver refuses it.
int encode_map_gate_up(CUtensorMap *map, const void *W1e, const void *W3e, int d, int ffn,
                       int *swapped);

}  // namespace moe
