// Grouped expert GEMMs on CTA pairs: a cluster of two CTAs on neighbouring
// SMs computes one 256-row x 256-column tile with tcgen05 .cta_group::2.
//
// Same operation and work units as gemm_tc.cu (gate/up with the SwiGLU
// epilogue, or the down projection), for the many-rows-per-expert regime:
//   - each CTA holds 128 token rows (A) and half of the 256 weight rows (B):
//     for gate/up CTA 0 holds the W1 rows and CTA 1 the W3 rows of the same
//     128 features, for down each holds 128 of the 256 output rows;
//   - the even CTA issues the MMAs; the tensor cores read A and B from both
//     CTAs' shared memory and each CTA's tensor memory receives its own 128
//     rows of the fp32 accumulator.
// Per CTA and 64-deep contraction step that is 32 KB of operands instead of
// 48 KB for a single-CTA 128 x 256 tile, so six pipeline stages fit in shared
// memory and each SM streams a third fewer bytes per FLOP.
//
// Barriers (same offsets in both CTAs):
//   full[s]      even CTA only: one arrival with the stage's byte count from
//                the even CTA's producer; both CTAs' TMA copies complete
//                bytes on it;
//   empty[s]     both CTAs: the even CTA's MMA commit multicasts to both;
//   acc_full[a]  both CTAs: MMA commit multicast, read by each epilogue;
//   acc_empty[a] even CTA only: one arrival per epilogue warp of both CTAs;
//   drain, bye   teardown: the MMA drain, and a pair handshake so neither CTA
//                leaves while the other may still touch its shared memory.
// Every wait is bounded as in gemm_tc.cu.
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kPairM = 256;
constexpr int kHalfM = 128;
constexpr int kNB = 256;
constexpr int kHalfN = 128;
constexpr int kStages = 6;
constexpr int kMaxE = MOE_MAX_EXPERTS;
constexpr int kThreads = 192;
constexpr int kABytes = kHalfM * 128;
constexpr int kBBytes = kHalfN * 128;
constexpr int kRing = kStages * (kABytes + kBBytes);
constexpr int kBars = (2 * kStages + 6) * 8;
constexpr int kMisc = 16 + 4 * (3 * kMaxE + 2);
constexpr size_t kSmem = 1024 + kRing + kBars + kMisc;
constexpr uint32_t kTmemCols = 2 * kNB;
constexpr int kAccEmptyArrivals = 8;  // lane 0 of the 4 epilogue warps of each CTA
constexpr uint16_t kBothCtas = 0x3;

struct PairArgs {
    CUtensorMap mapA;          // token rows [rows][K] bf16, box {64, 128}
    CUtensorMap mapB0[kMaxE];  // W1[e] (gate/up) or W2[e] (down): [N][K], box {64, 128}
    CUtensorMap mapB1[kMaxE];  // W3[e] (gate/up only)
    const int *offsets;        // [E + 1]
    void *out;                 // h bf16 [rows][N]  or  y fp32 [splits][rows][N]
    int *status;
    unsigned long long wait_limit_ns;
    int E, rows, K, N, kblocks, kps, splits;
};

struct PairUnit {
    int e, row0, nrows, n0, ks, kb0, kb1;  // row0 / nrows: the pair's 256-row tile
};

__device__ __forceinline__ PairUnit decode_pair_unit(int u, const int *s_off, const int *s_mt,
                                                     const int *s_ustart, const PairArgs &a,
                                                     int NOUT) {
    int e = 0;
    while (e + 1 < a.E && u >= s_ustart[e + 1]) ++e;
    const int local = u - s_ustart[e];
    const int mtn = s_mt[e];
    const int mt = local % mtn;
    const int rest = local / mtn;
    PairUnit w;
    w.e = e;
    w.ks = rest % a.splits;
    w.n0 = (rest / a.splits) * NOUT;
    w.row0 = s_off[e] + mt * kPairM;
    w.nrows = min(kPairM, s_off[e + 1] - w.row0);
    w.kb0 = w.ks * a.kps;
    w.kb1 = min(w.kb0 + a.kps, a.kblocks);
    return w;
}

template <bool SWIGLU>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    grouped_gemm_pair(const __grid_constant__ PairArgs a) {
    constexpr int NOUT = SWIGLU ? kHalfN : kNB;
    constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kPairM, kNB);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + kStages * kABytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kRing);
    uint64_t *empty = full + kStages;
    uint64_t *acc_full = empty + kStages;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint64_t *bye = drain + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bye + 1);
    volatile int *s_abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *s_bye_ok = reinterpret_cast<volatile int *>(tmem_slot + 2);
    int *s_off = reinterpret_cast<int *>(tmem_slot + 4);  // [kMaxE + 1]
    int *s_mt = s_off + kMaxE + 1;                         // [kMaxE]
    int *s_ustart = s_mt + kMaxE;                          // [kMaxE + 1]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool even = rank == 0;
    const int E = a.E;
    const int NT = (a.N + NOUT - 1) / NOUT;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&acc_full[i], 1);
            ptx::mbar_init(&acc_empty[i], kAccEmptyArrivals);
        }
        ptx::mbar_init(drain, 1);
        ptx::mbar_init(bye, 1);
        *s_abort = 0;
        *s_bye_ok = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(tmem_slot, kTmemCols);
        ptx::tmem_relinquish_pair();
    }
    if (warp == 0 && lane == 0) ptx::prefetch_tensormap(&a.mapA);
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x <= E) s_off[threadIdx.x] = a.offsets[threadIdx.x];
    ptx::tc_fence_before_sync();
    __syncthreads();
    // both CTAs' barriers are initialised before either signals the other's
    ptx::cluster_sync_all();
    ptx::tc_fence_after_sync();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int e = 0; e < E; ++e) {
            const int cnt = s_off[e + 1] - s_off[e];
            const int mt = cnt > 0 ? (cnt + kPairM - 1) / kPairM : 0;
            s_mt[e] = mt;
            s_ustart[e] = acc;
            acc += mt * NT * a.splits;
        }
        s_ustart[E] = acc;
    }
    __syncthreads();
    const uint32_t tmem_base = *tmem_slot;
    const int total = s_ustart[E];
    const int first = static_cast<int>(ptx::cluster_id_x());
    const int stride = static_cast<int>(ptx::cluster_count_x());

    if (warp == 0) {
        // ------------------------------------------------------------ producers
        if (lane == 0) {
            const uint32_t full0 = ptx::map_to_rank(ptx::smem_addr(&full[0]), 0);
            const uint32_t tx_bytes = 2u * (kABytes + kBBytes);
            int stage = 0;
            uint32_t ph = 0;
            int issued = 0;
            bool ok = true;
            for (int u = first; ok && u < total; u += stride) {
                const PairUnit w = decode_pair_unit(u, s_off, s_mt, s_ustart, a, NOUT);
                const CUtensorMap *mb =
                    (SWIGLU && !even) ? &a.mapB1[w.e] : &a.mapB0[w.e];
                const int brow = SWIGLU ? w.n0 : w.n0 + static_cast<int>(rank) * kHalfN;
                const int arow = w.row0 + static_cast<int>(rank) * kHalfM;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!ptx::mbar_wait_bounded(&empty[stage], ph ^ 1u, s_abort, a.status,
                                                kStatusProducerWait, a.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    if (even) ptx::mbar_arrive_expect_tx(&full[stage], tx_bytes);
                    const uint32_t fb = full0 + static_cast<uint32_t>(stage) * 8u;
                    ptx::tma_load_2d_pair(sA + stage * kABytes, &a.mapA, kb * kBlockK, arow, fb);
                    ptx::tma_load_2d_pair(sB + stage * kBBytes, mb, kb * kBlockK, brow, fb);
                    ++issued;
                    if (++stage == kStages) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (*s_abort && even) {
                // let both CTAs' copies in flight land (they count on full[])
                for (int i = 0; i < kStages && i < issued; ++i) {
                    if (stage == 0) {
                        stage = kStages - 1;
                        ph ^= 1u;
                    } else {
                        --stage;
                    }
                    ptx::mbar_wait_bounded(&full[stage], ph, nullptr, a.status, kStatusDrainWait,
                                           a.wait_limit_ns);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && even) {
            int stage = 0;
            uint32_t ph = 0;
            int it = 0;
            bool ok = true;
            for (int u = first; ok && u < total; u += stride, ++it) {
                const PairUnit w = decode_pair_unit(u, s_off, s_mt, s_ustart, a, NOUT);
                const int acc = it & 1;
                const uint32_t aph = static_cast<uint32_t>(it >> 1) & 1u;
                if (!ptx::mbar_wait_bounded(&acc_empty[acc], aph ^ 1u, s_abort, a.status,
                                            kStatusMmaWait, a.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kNB);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!ptx::mbar_wait_bounded(&full[stage], ph, s_abort, a.status,
                                                kStatusMmaWait, a.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint32_t a0 = ptx::smem_addr(sA + stage * kABytes);
                    const uint32_t b0 = ptx::smem_addr(sB + stage * kBBytes);
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk) {
                        ptx::mma_bf16_pair(d_tmem, ptx::desc_kmajor_sw128(a0 + kk * 32),
                                           ptx::desc_kmajor_sw128(b0 + kk * 32), kIdesc,
                                           (kb > w.kb0 || kk > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit_pair_multicast(&empty[stage], kBothCtas);
                    if (++stage == kStages) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit_pair_multicast(&acc_full[acc], kBothCtas);
            }
            ptx::mma_commit_pair(drain);
            ptx::mbar_wait_bounded(drain, 0, nullptr, a.status, kStatusDrainWait,
                                   a.wait_limit_ns);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;  // tensor-memory lanes 32*quad .. +31
        const int r = quad * 32 + lane;
        const uint32_t acc_empty0 = ptx::map_to_rank(ptx::smem_addr(&acc_empty[0]), 0);
        int it = 0;
        for (int u = first; u < total; u += stride, ++it) {
            const PairUnit w = decode_pair_unit(u, s_off, s_mt, s_ustart, a, NOUT);
            const int acc = it & 1;
            const uint32_t aph = static_cast<uint32_t>(it >> 1) & 1u;
            if (!ptx::mbar_wait_bounded(&acc_full[acc], aph, s_abort, a.status,
                                        kStatusEpilogueWait, a.wait_limit_ns))
                break;
            ptx::tc_fence_after_sync();
            const int hrow0 = w.row0 + static_cast<int>(rank) * kHalfM;
            const int hrows = max(0, min(kHalfM, w.nrows - static_cast<int>(rank) * kHalfM));
            const uint32_t tb = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                static_cast<uint32_t>(acc * kNB);
            if (quad * 32 < hrows) {
                const bool row_ok = r < hrows;
                if (SWIGLU) {
                    __nv_bfloat16 *hrow =
                        static_cast<__nv_bfloat16 *>(a.out) + (size_t)(hrow0 + r) * a.N + w.n0;
#pragma unroll 1
                    for (int c = 0; c < kHalfN; c += 32) {
                        uint32_t U[32], V[32];
                        ptx::tmem_ld_32x32b_x32(tb + c, U);
                        ptx::tmem_ld_32x32b_x32(tb + kHalfN + c, V);
                        ptx::tmem_ld_wait();
                        if (row_ok && w.n0 + c < a.N) {
                            uint32_t packed[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const float u0 = __uint_as_float(U[2 * i]);
                                const float u1 = __uint_as_float(U[2 * i + 1]);
                                const float v0 = __uint_as_float(V[2 * i]);
                                const float v1 = __uint_as_float(V[2 * i + 1]);
                                const float h0 = u0 / (1.f + expf(-u0)) * v0;
                                const float h1 = u1 / (1.f + expf(-u1)) * v1;
                                const __nv_bfloat162 p = __floats2bfloat162_rn(h0, h1);
                                packed[i] = *reinterpret_cast<const uint32_t *>(&p);
                            }
                            uint4 *dst = reinterpret_cast<uint4 *>(hrow + c);
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1],
                                                    packed[4 * q + 2], packed[4 * q + 3]);
                        }
                    }
                } else {
                    float *yrow = static_cast<float *>(a.out) +
                                  ((size_t)w.ks * a.rows + hrow0 + r) * a.N + w.n0;
#pragma unroll 1
                    for (int c = 0; c < kNB; c += 32) {
                        uint32_t Y[32];
                        ptx::tmem_ld_32x32b_x32(tb + c, Y);
                        ptx::tmem_ld_wait();
                        if (row_ok && w.n0 + c < a.N) {
                            float4 *dst = reinterpret_cast<float4 *>(yrow + c);
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                dst[q] = make_float4(__uint_as_float(Y[4 * q]),
                                                     __uint_as_float(Y[4 * q + 1]),
                                                     __uint_as_float(Y[4 * q + 2]),
                                                     __uint_as_float(Y[4 * q + 3]));
                        }
                    }
                }
            }
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(acc_empty0 + static_cast<uint32_t>(acc) * 8u);
        }
    }

    // Teardown: neither CTA leaves (and frees tensor memory) before the other
    // is done with the pair's shared memory and barriers.
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0) {
        ptx::mbar_arrive_cluster(ptx::map_to_rank(ptx::smem_addr(bye), rank ^ 1u));
        *s_bye_ok = ptx::mbar_wait_bounded(bye, 0, nullptr, a.status, kStatusDrainWait,
                                           a.wait_limit_ns)
                        ? 1
                        : 0;
    }
    __syncthreads();
    if (warp == 1 && *s_bye_ok) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

std::mutex g_pair_mutex;

template <bool SWIGLU>
int run_pair(PairArgs &args, int units_bound, cudaStream_t s) {
    auto kernel = grouped_gemm_pair<SWIGLU>;
    static bool attr_set[64];
    static int max_pairs[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
    {
        std::lock_guard<std::mutex> g(g_pair_mutex);
        if (!attr_set[dev]) {
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kSmem)) != cudaSuccess)
                return MOE_ERR_CUDA;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2 * (device_sm_count() / 2));
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = kSmem;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0)
                n = device_sm_count() / 2;
            (void)cudaGetLastError();
            max_pairs[dev] = n;
            attr_set[dev] = true;
        }
    }
    int pairs = units_bound < max_pairs[dev] ? units_bound : max_pairs[dev];
    if (pairs <= 0) return MOE_OK;
    return launch_pdl(kernel, dim3(2 * pairs), kThreads, kSmem, s, args) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

int fill_pair(PairArgs &args, const void *A, const int *offsets, void *out, int rows, int K, int N,
              int E) {
    args.offsets = offsets;
    args.out = out;
    args.E = E;
    args.rows = rows;
    args.K = K;
    args.N = N;
    args.kblocks = (K + kBlockK - 1) / kBlockK;
    args.wait_limit_ns = kWaitLimitNs;
    args.status = device_status_ptr();
    if (args.status == nullptr) return MOE_ERR_CUDA;
    return encode_map_bf16_2d(&args.mapA, A, K, rows, kBlockK, kHalfM);
}

}  // namespace

size_t pair_gemm_smem_bytes() { return kSmem; }

int launch_swiglu_pair(const void *x_perm, const int *offsets, const void *const *W1,
                       const void *const *W3, int rows, int d, int ffn, int E, void *h,
                       cudaStream_t s) {
    if (rows == 0) return MOE_OK;
    PairArgs args;
    int rc = fill_pair(args, x_perm, offsets, h, rows, d, ffn, E);
    if (rc != MOE_OK) return rc;
    for (int e = 0; e < E; ++e) {
        if ((rc = encode_map_bf16_2d(&args.mapB0[e], W1[e], d, ffn, kBlockK, kHalfN)) != MOE_OK)
            return rc;
        if ((rc = encode_map_bf16_2d(&args.mapB1[e], W3[e], d, ffn, kBlockK, kHalfN)) != MOE_OK)
            return rc;
    }
    args.splits = 1;
    args.kps = args.kblocks;
    const int NT = (ffn + kHalfN - 1) / kHalfN;
    const int units_bound = ((rows + kPairM - 1) / kPairM + E) * NT;
    return run_pair<true>(args, units_bound, s);
}

int launch_down_pair(const void *h, const int *offsets, const void *const *W2, int rows, int d,
                     int ffn, int E, int splits, int kps, float *y, cudaStream_t s) {
    if (rows == 0) return MOE_OK;
    PairArgs args;
    int rc = fill_pair(args, h, offsets, y, rows, ffn, d, E);
    if (rc != MOE_OK) return rc;
    for (int e = 0; e < E; ++e)
        if ((rc = encode_map_bf16_2d(&args.mapB0[e], W2[e], ffn, d, kBlockK, kHalfN)) != MOE_OK)
            return rc;
    args.splits = splits;
    args.kps = kps;
    const int NT = (d + kNB - 1) / kNB;
    const int units_bound = ((rows + kPairM - 1) / kPairM + E) * NT * splits;
    return run_pair<false>(args, units_bound, s);
}

}  // namespace moe
