/*
 * moe.h -- C ABI of libmoe.so: the Mixtral sparse mixture-of-experts
 * feed-forward layer on an NVIDIA B300 (sm_103a).
 *
 * The layer (sources named by page title and passage):
 *   - Router: a linear layer, logits = x . W_g, one score per expert; the two
 *     largest are kept, the others are set to -inf, and a softmax over the
 *     kept scores gives the gates ("Mixtral of Experts" (azimuth.plus),
 *     router paragraph; two experts per token: "Mixtral of Experts"
 *     (tellworld.net), "How Mixtral 8x7B is built").
 *   - Experts: each a SwiGLU feed-forward network with its own weights
 *     ("Mixtral of Experts" (azimuth.plus), expert paragraph) -- gate, up and
 *     down projections 4096 -> 14336 -> 4096 ("Mixtral > Architecture
 *     Overview", parameter-count paragraph):
 *        y_e(x) = W2[e] . ( silu(W1[e] . x) * (W3[e] . x) ),  silu(u) = u/(1+e^-u).
 *   - Only the chosen experts run; their outputs are summed weighted by the
 *     gates ("Mixtral & Sparse MoE (2024) > The Solution", routing paragraph;
 *     "Mixtral" curriculum page, flow "scores experts -> run chosen MLPs ->
 *     weighted expert outputs"):
 *        out[t] = sum_j gates[t][j] * y_{idx[t][j]}(x[t]).
 *   - Every token is independent of every other ("Mixtral > Architecture
 *     Overview", paragraph on sparse feed-forward computation).
 *
 * Readings where the pages are silent: ties between equal logits go to the
 * lower expert index and slot 0 holds the larger logit; W1 is the gate and W3
 * the up projection; silu has beta = 1; the router has no bias (the optional
 * per-expert bias is added to the fp32 logits before selection, for skewed
 * benchmarks); every token's k rows are computed (no capacity limit).
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers owned by the caller, unless the name
 *     says host.  The weight-pointer arrays W1/W3/W2 are HOST arrays of E
 *     device pointers, read during the call only.
 *   - Layouts are row-major and dense:
 *       x, out  [T][d]          W_g [E][d]
 *       W1[e], W3[e] [ffn][d]   (row c = input weights of hidden feature c)
 *       W2[e]   [d][ffn]        (row n = input weights of output feature n)
 *     In the pages' row-vector notation x.W1 this is W1 . x here.
 *   - dtype MOE_BF16: x, W_g, W1/W3/W2, out are bf16; router logits, gates and
 *     every accumulation are fp32; the expert hidden activation h is stored
 *     as bf16 and the expert outputs as fp32.  MOE_F32: everything fp32, with
 *     plain fp32 FMAs (never TF32).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without synchronising.  Arguments are
 *     validated on the host before anything is enqueued; on any error nothing
 *     is launched.  Faults inside kernels surface at the caller's next
 *     synchronisation; bounded waits inside the kernels that expire set a
 *     device status word read by moe_device_status().
 *   - The library allocates no device memory: scratch comes from the caller's
 *     `workspace` (size from moe_workspace_bytes, 256-byte aligned).  Calls on
 *     different streams need different workspaces.
 *   - Launch graphs (moe_forward, moe_forward_ex, moe_block_forward,
 *     moe_forward_host_io): the second call with exactly the same arguments
 *     (every pointer, size, option and the tile plan) captures its launches
 *     into a CUDA graph on a private stream, and that call and later ones
 *     with the same arguments launch the graph on `stream`: the same kernels
 *     with the same parameters, so the same bits.  The library keeps those
 *     graphs, and the pointers inside them, for up to 64 argument sets per
 *     process (a new set replaces the least recently used one); a graph only
 *     runs for a call that passes the same pointers again, and reads the
 *     buffers' contents as they are then.  moe_graph_cache_stats reports how
 *     often calls were served from the cache.  A call on a
 *     stream that is being captured enqueues its kernels directly, into the
 *     caller's graph.  MOE_GRAPHS=0 in the environment turns graphs off.
 *   - Limits: 1 <= E <= 64, 1 <= k <= min(E, 8), T >= 0 (T = 0 is a no-op).
 *     ("Mixtral > Architecture Overview" weighs 4 or 64 experts against 8;
 *     Mixtral itself uses E = 8, k = 2.)  bf16 needs
 *     d and ffn multiples of 64 and 16-byte aligned tensors; fp32 needs d a
 *     multiple of 4.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_ARG = -1,         /* null pointer, negative size, k > E, ...       */
    MOE_ERR_UNSUPPORTED = -2, /* E > 64, k > 8, alignment or shape limits      */
    MOE_ERR_WORKSPACE = -3,   /* workspace missing, too small or misaligned    */
    MOE_ERR_CUDA = -4,        /* a CUDA runtime call or launch failed          */
    MOE_ERR_DEVICE = -5       /* a kernel's bounded wait expired (status word) */
} moe_status;

#define MOE_MAX_EXPERTS 64
#define MOE_MAX_TOPK 8

/*
 * Routing options (moe_forward_ex, moe_route_from_logits_ex).  A NULL
 * options pointer, or all fields zero, is the layer as "Mixtral of Experts"
 * (azimuth.plus, router paragraph) states it.
 *   gating: MOE_GATING_TOPK_SOFTMAX -- keep the top k logits, softmax over
 *     them (the gates sum to 1); MOE_GATING_SOFTMAX_TOPK -- softmax over all E
 *     logits, keep the k largest probabilities as they are, not renormalised
 *     (a reading of "Mixtral & Sparse MoE (2024) > The Solution", routing
 *     paragraph).
 *   capacity: the most (token, slot) selections each expert keeps; an expert
 *     keeps its first `capacity` selections in token order and drops the rest
 *     ("The Solution", load-balancing paragraph: capacity constraints).
 *     <= 0: no limit.  moe_capacity() gives ceil(factor * T * k / E).
 *   drop_policy: what a dropped selection's gate does.  MOE_DROP_LOSE -- its
 *     mass is lost (the token's output is the kept slots' weighted sum);
 *     MOE_DROP_RENORMALIZE -- the token's kept gates are scaled to sum to its
 *     full gate mass (a token with every slot dropped gets zero output).
 */
typedef enum { MOE_GATING_TOPK_SOFTMAX = 0, MOE_GATING_SOFTMAX_TOPK = 1 } moe_gating;
typedef enum { MOE_DROP_LOSE = 0, MOE_DROP_RENORMALIZE = 1 } moe_drop_policy;
typedef struct {
    int gating;      /* moe_gating      */
    int capacity;    /* rows per expert */
    int drop_policy; /* moe_drop_policy */
} moe_options;

/* Text for a status code (static storage). */
const char *moe_strerror(int status);

/* Library version, e.g. 100 = 0.1.0. */
int moe_version(void);

/* Scratch bytes moe_forward needs for this shape; written to *bytes.
 * Returns MOE_OK or an argument error. */
int moe_workspace_bytes(int T, int d, int ffn, int E, int k, int dtype, size_t *bytes);

/*
 * The whole layer: out = MoE(x).  Runs the router, the grouping by expert,
 * the two grouped expert GEMMs and the gated combine on `stream`.
 *   router_bias: NULL or a device fp32 [E] added to the logits.
 *   workspace: device scratch of at least moe_workspace_bytes(...) bytes.
 */
int moe_forward(const void *x, const void *W_g, const float *router_bias,
                const void *const *W1, const void *const *W3, const void *const *W2,
                int T, int d, int ffn, int E, int k, int dtype, void *out,
                void *workspace, size_t workspace_bytes, void *stream);

/*
 * moe_forward with routing options (see moe_options; NULL = moe_forward).
 * The expert GEMMs only see the kept rows, so a capacity limit also removes
 * the dropped rows' work.
 */
int moe_forward_ex(const void *x, const void *W_g, const float *router_bias,
                   const void *const *W1, const void *const *W3, const void *const *W2,
                   int T, int d, int ffn, int E, int k, int dtype, const moe_options *options,
                   void *out, void *workspace, size_t workspace_bytes, void *stream);

/*
 * One pre-norm MoE block of a decoder layer, in place on the residual stream
 * x [T][d]:
 *     x <- round(x + MoE(RMSNorm(x))),   RMSNorm(x) = x / sqrt(mean(x^2) + eps)
 * with gain 1 (each feed-forward sub-block of the Mistral decoder is
 * pre-normalised and added back to the residual stream: "Mixtral of Experts"
 * (azimuth.plus), decoder paragraph).  Gives the same bits as
 * moe_add_rmsnorm(x, NULL, xn), moe_forward_ex(xn, ..., out),
 * moe_add_rmsnorm(x, out, xn): the RMSNorm is done inside the router and the
 * grouping pass (the normalised rows are never stored) and the residual add
 * inside the combine, which saves one kernel and 3 T d elements of HBM
 * traffic per block.  Arguments as moe_forward_ex; the workspace size is
 * moe_workspace_bytes(...); eps >= 0.
 */
int moe_block_forward(void *x, const void *W_g, const float *router_bias,
                      const void *const *W1, const void *const *W3, const void *const *W2,
                      int T, int d, int ffn, int E, int k, int dtype, float eps,
                      const moe_options *options, void *workspace, size_t workspace_bytes,
                      void *stream);

/*
 * Backward of the layer, for training ("Mixtral & Sparse MoE (2024) > The
 * Solution" and "Mixtral of Experts" (azimuth.plus) describe training the
 * model; no page prints the backward, which is the chain rule through the
 * forward above).  For the upstream gradient d_out [T][d] (dtype) of the
 * layer output it writes, overwriting:
 *   d_x   [T][d] dtype          gradient of x (rounded once);
 *   d_W_g [E][d] fp32           gradient of the router matrix;
 *   d_W1[e], d_W3[e] [ffn][d] fp32 and d_W2[e] [d][ffn] fp32 (host arrays of E
 *   device pointers, 16-byte aligned).
 * Which experts a token picks is piecewise constant in the inputs, so no
 * gradient flows through the choice; the softmax over the kept logits is
 * differentiated.  Routing and the gate/up projections are recomputed from x,
 * so nothing from a forward call has to be kept.  Every sum runs in a fixed
 * order (no atomics): the gradients are deterministic.  Limits: dtype MOE_BF16
 * (fp32 gives MOE_ERR_UNSUPPORTED) and the default routing (top-k softmax, no
 * capacity limit).  router_bias may be NULL.  workspace: at least
 * moe_backward_workspace_bytes(...) bytes, 256-byte aligned.
 */
int moe_backward_workspace_bytes(int T, int d, int ffn, int E, int k, int dtype, size_t *bytes);
int moe_backward(const void *x, const void *W_g, const float *router_bias,
                 const void *const *W1, const void *const *W3, const void *const *W2,
                 int T, int d, int ffn, int E, int k, int dtype, const void *d_out, void *d_x,
                 float *d_W_g, float *const *d_W1, float *const *d_W3, float *const *d_W2,
                 void *workspace, size_t workspace_bytes, void *stream);

/* Capacity for a capacity factor: ceil(factor * T * k / E), written to
 * *capacity (factor <= 0 gives 0, i.e. no limit). */
int moe_capacity(double capacity_factor, int T, int k, int E, int *capacity);

/*
 * Same as moe_forward, with the tokens and the result in HOST memory: copies
 * x_host -> x_dev, runs the layer, and delivers the result to out_host, all
 * enqueued on `stream`.  When out_host is page-locked (pinned or registered)
 * host memory, the layer's last kernel writes the result there directly and
 * out_dev is not used; otherwise the layer writes out_dev and a copy
 * out_dev -> out_host follows.  Likewise, for batches the router takes in
 * one pass (bf16, up to 8 experts, fewer than 1536 tokens) a page-locked
 * x_host is read by the router directly, which leaves the rows in x_dev for
 * the later kernels; other batches copy x_host -> x_dev first.  The caller
 * synchronises the stream before reading out_host, and keeps x_host unchanged
 * until then.
 */
int moe_forward_host_io(const void *x_host, void *out_host, void *x_dev, void *out_dev,
                        const void *W_g, const float *router_bias,
                        const void *const *W1, const void *const *W3,
                        const void *const *W2, int T, int d, int ffn, int E, int k,
                        int dtype, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Router stage: logits [T][E] fp32 (x . W_g + bias, fp32 accumulation),
 * idx [T][k] int32 (slot 0 = larger logit, ties to the lower index),
 * gates [T][k] fp32 (softmax over the k kept logits).
 */
int moe_router(const void *x, const void *W_g, const float *router_bias, int T, int d,
               int E, int k, int dtype, float *logits, int *idx, float *gates,
               void *stream);

/* Scratch bytes for moe_route_from_logits. */
int moe_route_workspace_bytes(int T, int E, int k, size_t *bytes);

/*
 * Selection and grouping from given fp32 logits [T][E]:
 *   idx, gates as in moe_router;
 *   counts [E]: rows routed to each expert; offsets [E+1]: exclusive prefix
 *   sum (offsets[E] = T*k);
 *   perm [T*k]: row r of the expert-grouped order holds (token t, slot j) as
 *   t*k + j, rows of one expert in ascending token order;
 *   inv [T*k]: inv[t*k + j] = r.
 * Deterministic: identical logits give bit-identical outputs.
 */
int moe_route_from_logits(const float *logits, int T, int E, int k, int *idx,
                          float *gates, int *counts, int *offsets, int *perm, int *inv,
                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * moe_route_from_logits with routing options: gates follow options->gating;
 * with a capacity only kept selections get rows -- counts are the kept
 * counts, perm holds offsets[E] entries and inv[t*k + j] is -1 for a dropped
 * selection.  gates are the routing gates before any drop.
 */
int moe_route_from_logits_ex(const float *logits, int T, int E, int k,
                             const moe_options *options, int *idx, float *gates, int *counts,
                             int *offsets, int *perm, int *inv, void *workspace,
                             size_t workspace_bytes, void *stream);

/*
 * Gather: x_perm[r] = x[perm[r] / k] for r < rows (exact copies); rows <= T*k
 * (T*k without a capacity limit, offsets[E] with one).
 */
int moe_permute(const void *x, const int *perm, int rows, int T, int d, int k, int dtype,
                void *x_perm, void *stream);

/*
 * Grouped gate/up projections with the SwiGLU product, for rows grouped by
 * expert (rows offsets[e] .. offsets[e+1]-1 belong to expert e):
 *   h[r][c] = silu(sum_i x_perm[r][i] W1[e][c][i]) * (sum_i x_perm[r][i] W3[e][c][i])
 * x_perm [rows][d], h [rows][ffn] (dtype), offsets device int32 [E+1].
 * bf16 runs on the tcgen05 tensor cores (fp32 accumulation in tensor memory);
 * fp32 on plain FMAs.
 */
int moe_expert_swiglu(const void *x_perm, const int *offsets, const void *const *W1,
                      const void *const *W3, int rows, int d, int ffn, int E, int dtype,
                      void *h, void *stream);

/* Split count moe_expert_down uses for this shape (>= 1); written to *splits. */
int moe_down_splits(int T, int d, int ffn, int E, int k, int dtype, int *splits);

/*
 * Grouped down projection: y[s][r][n] = sum_{c in split s} h[r][c] W2[e][n][c],
 * fp32 partial sums [splits][rows][d], splits from moe_down_splits(T, ...)
 * with rows = T*k.  The full y is the sum over s (taken in moe_combine).
 */
int moe_expert_down(const void *h, const int *offsets, const void *const *W2, int T,
                    int d, int ffn, int E, int k, int dtype, float *y_partial,
                    void *stream);

/*
 * Gated combine: out[t][n] = sum_j gates[t][j] * (sum_s y[s][inv[t*k+j]][n]),
 * fp32 sums in fixed order, one rounding to dtype.  Slots with inv < 0 (dropped
 * by a capacity limit) are skipped; moe_forward_ex's renormalising drop policy
 * is applied inside moe_forward_ex, not by this entry point.
 */
int moe_combine(const float *y_partial, int splits, const float *gates, const int *inv,
                int T, int d, int k, int dtype, void *out, void *stream);

/*
 * Stacked-layer helper (not part of the layer itself): if `add` is not NULL,
 * x <- round(x + add) in place; then xn = x / sqrt(mean(x^2) + eps) with
 * gain 1 (RMSNorm before each feed-forward sub-block of a Mistral decoder,
 * "Mixtral of Experts" (azimuth.plus), decoder paragraph).  [T][d], dtype;
 * d * element size a multiple of 16 bytes and 16-byte aligned tensors.  The
 * sum of squares is taken in the order moe_block_forward's fused RMSNorm
 * uses, so both give the same bits.
 */
int moe_add_rmsnorm(void *x, const void *add, void *xn, int T, int d, float eps,
                    int dtype, void *stream);

/*
 * Device status word: synchronises `stream`, writes the word to *status
 * (0 = no kernel reported a problem; otherwise the code of the first expired
 * bounded wait) and clears it if `clear` is non-zero.
 */
int moe_device_status(void *stream, int *status, int clear);

/*
 * Self-test of the bounded-wait path: launches one tiny kernel that waits on
 * a barrier nothing arrives at, with the given limit in nanoseconds (clamped
 * to 1 us .. 100 ms); it gives up, records the expiry in the status word and
 * returns, leaving the context usable.
 */
int moe_selftest_wait_timeout(unsigned int limit_ns, void *stream);

/* Number of kernels moe_forward launches for this shape (for launch counts). */
int moe_forward_launches(int T, int d, int ffn, int E, int k, int dtype, int *launches);

/*
 * Counters of the launch-graph cache (see "Launch graphs" above), for all
 * devices of the process since load or the last reset:
 *   entries       argument sets held now (at most 64);
 *   replays       calls served by launching a cached graph;
 *   captures      graphs captured (the second call of an argument set);
 *   direct_calls  calls that enqueued their kernels one by one (first call of
 *                 an argument set, graphs off, a capturing caller stream, or a
 *                 failed capture);
 *   evictions     argument sets dropped, least recently used first, to make
 *                 room for a new one.
 * A serving loop whose pointers or sizes change every call shows replays near
 * zero: the cache is not helping it (MOE_GRAPHS=0 turns it off).
 * reset != 0 zeroes the four counts after reading them.  No device work.
 */
typedef struct {
    long long entries, replays, captures, direct_calls, evictions;
} moe_graph_stats;
int moe_graph_cache_stats(moe_graph_stats *stats, int reset);

/*
 * The pages have no counterpart to this entry point: it is a convenience for
 * callers that cannot allocate device memory where they run the layer (an
 * inference-engine plugin handed fixed buffers that must not allocate in its
 * enqueue step, a serving process whose memory budget was reserved at
 * start-up).  Its kernels are enqueued directly on `stream` (the launch
 * graphs described above are not used by this entry point).
 *
 * Same result as moe_forward, but the scratch is a fixed array of
 * MOE_STATIC_SCRATCH_BYTES inside the library on each device, held until the
 * process exits, so no workspace is passed and nothing is allocated.  The
 * caller still passes x, the weights and out.
 *   - Shapes whose moe_workspace_bytes(...) exceeds MOE_STATIC_SCRATCH_BYTES
 *     are rejected with MOE_ERR_WORKSPACE before anything is enqueued.  At
 *     the Mixtral shape (d = 4096, ffn = 14336, 8 experts, top-2) every
 *     batch of up to 81 tokens fits.  Whether a batch fits depends on its
 *     tile plan (the token tile height and the down projection's split
 *     change with T), so it is not monotone in T (some larger batches fit
 *     too): check moe_workspace_bytes(...) <= MOE_STATIC_SCRATCH_BYTES.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture begins.
 *   - Every call on a device shares the one array: calls whose GPU work can
 *     overlap (other streams, other host threads) race and must be
 *     serialised by the caller.  Contents left by a previous call are never
 *     read; nothing needs clearing.
 */
#define MOE_STATIC_SCRATCH_BYTES (16u << 20)
int moe_forward_static_scratch(const void *x, const void *W_g, const float *router_bias,
                               const void *const *W1, const void *const *W3,
                               const void *const *W2, int T, int d, int ffn, int E, int k,
                               int dtype, void *out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
